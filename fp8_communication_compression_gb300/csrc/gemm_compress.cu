// The tensor-core GEMM whose epilogue compresses or quantises its fp32
// result before it leaves the SM.
//
// AGoQ (gist.science summary of arXiv 2605.00539), 2.C: the quantisation
// runs inside the adjacent GEMM kernel, the tensor cores doing the matrix
// product and the CUDA cores the quantisation.  One kernel, three
// epilogues:
//  * TACO's compressor (gist.science summary of arXiv 2604.24088,
//    2.B.1-2.B.3): the partial sum Y = A B^T of a row-parallel layer leaves
//    the kernel already as ASH + DS E4M3 codes with their two scalars per
//    block, ready for the two-shot exchange, instead of being written in
//    bf16 and read back by the compressor;
//  * AGoQ 2.B's accumulation of a weight gradient into the FP8 main
//    gradient (dequantise, add, requantise, in place);
//  * AGoQ 2.A's block-wise LAAQ quantisation of an activation (4, 5, 6 or 8
//    bits a code, packed).
//
// Design (sm_103a):
//  * A persistent grid, one CTA per SM, walks the 128 x 256 tiles of Y
//    (128 x 128 where N % 256 != 0) in turn.  Warp 0 is the TMA producer:
//    it streams 128 x 64 tiles of A and 256 x 64 tiles of B (bf16, 128-byte
//    swizzle) through a 4-stage mbarrier ring, from one output tile into
//    the next without a gap.  Warp 1 allocates 512 columns of tensor memory
//    (two fp32 accumulators of 256 columns) and one of its threads issues
//    the tcgen05.mma steps (128 x 256 x 16 each, four per 64-wide stage),
//    frees each stage with tcgen05.commit, and signals a finished
//    accumulator the same way.  Warps 2-5 are the epilogue: while they
//    process tile i from one accumulator, the MMAs of tile i + 1 fill the
//    other.
//  * The accumulator's lane is the tile row, so after tcgen05.ld each
//    epilogue thread holds 128 consecutive fp32 values of one row: exactly
//    one block, the layout the stand-alone codec kernels give a thread.
//    The block's arithmetic (the 128-point Walsh-Hadamard transform, alpha,
//    s and E4M3; or the FP8 accumulation; or the LAAQ quantisation) runs in
//    that thread's registers, and the codes go through the warp's staging
//    rows and TMA stores.
//  * Split tail: when the tiles do not fill whole rounds of SMs and K is
//    long enough, the tiles of the last round are cut along K into 2-4
//    pieces dealt out like tiles; their fp32 partial sums meet in a
//    caller's workspace and the warp that stores a tile quarter's last
//    piece adds them up in piece order, then runs the epilogue (no spin
//    waits).
//  * Every mbarrier wait is time-limited; a wait that runs out sets a flag
//    readable through taco_device_error() and the CTA winds down.

#include <atomic>
#include <cfloat>

#include "codec_math.cuh"
#include "device_utils.cuh"
#include "internal.h"
#include "laaq_math.cuh"
#include "reduce_math.cuh"
#include "tcgen05.cuh"

namespace taco {

// Watchdog flags of this file's kernel (bit 5), read with the codec
// kernels' flags by taco_device_error().
__device__ unsigned int g_gemm_error;

namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kGThreads = 192;                  // warps: 0 producer, 1 MMA, 2-5 epilogue
constexpr uint32_t kABytes = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kErrGemm = 32u;

// Tile width BN (256, or 128 where 256-wide tiles would leave more SMs idle
// in the last round): stage and tensor-memory sizes follow from it.
template <int BN> struct GemmCfg {
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr uint32_t kBBytes = BN * kBK * 2;            // 32 or 16 KB
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;    // 48 or 32 KB
    static constexpr uint32_t kAccCols = BN;                      // fp32 accumulator, a column per tile column
    static constexpr uint32_t kTmemCols = 2 * BN;                 // two accumulators
    static constexpr int kBlocks = BN / 128;                      // compression blocks per tile row
    static constexpr uint32_t kStageOut = 4 * kBlocks * 4096;     // staging: 4 warps x blocks x 32 rows x 128 B
    static constexpr uint32_t kBars = 8 * (2 * kStages + 4);      // full / empty per stage and per accumulator
    static constexpr uint32_t kSmem = 1024 + kStages * kStageBytes + kStageOut + kBars + 16;
    static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
    static_assert(kSmem <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Compresses one 128-element block of the thread's row into the staging row
// at `orow` (swizzled), and returns its alpha and s.  load32(j, x) gives
// the block's values 32 j .. 32 j + 31 (from tensor memory, or the summed
// partials of a split tile).  y_row (optional) gets those values.
template <class Load>
__device__ __forceinline__ void compress_block(Load &&load32, float *y_row, uint32_t orow, uint32_t swz,
                                               float e_target, float eps, float &alpha, float &scale)
{
    float2 v[64];
    float2 acc[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float x[32];
        load32(j, x);
        if (y_row) {
            float4 *yo = reinterpret_cast<float4 *>(y_row + 32 * j);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                yo[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
        }
        // step 1 (energy) and the bit-0 butterfly stage of step 3
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const int kk = 16 * j + t;
            const float2 xx = make_float2(x[2 * t], x[2 * t + 1]);
            acc[kk & 7] = (kk < 8) ? __fmul2_rn(xx, xx) : __ffma2_rn(xx, xx, acc[kk & 7]);
            v[kk] = make_float2(xx.x + xx.y, xx.x - xx.y);
        }
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
            acc[i] = __fadd2_rn(acc[i], acc[i + w]);
    const float ss = acc[0].x + acc[0].y;
    // step 3: remaining butterflies; the last is fused with the scaling
    fwht128_upper_but_last(v);
    const float mh = max_abs_last_stage(v);
    // step 2: alpha = sqrt(E / (m + eps));  step 4: s = 448 / max|y|
    alpha = sqrtf(e_target / (ss * BlockConst<128>::inv_n + eps));
    const float ac = alpha * BlockConst<128>::c;
    const float M = ac * mh;
    scale = (M > 0.0f) ? fminf(448.0f / M, FLT_MAX) : 1.0f;
    float k = ac * scale;
    if (!(k <= FLT_MAX)) {  // block of tiny values: apply the two factors separately
        const float2 ac2 = make_float2(ac, ac);
#pragma unroll
        for (int i = 0; i < 64; ++i)
            v[i] = __fmul2_rn(v[i], ac2);
        k = scale;
    }
    last_stage_scaled(v, make_float2(k, k));
    // step 5: E4M3 codes into the swizzled staging row
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t w0, w1, w2, w3;
        encode8_prescaled(&v[8 * j], w0, w1);
        encode8_prescaled(&v[8 * j + 4], w2, w3);
        sts128(orow + ((static_cast<uint32_t>(j) << 4) ^ swz), w0, w1, w2, w3);
    }
}

// AGoQ 2.B local accumulation of one 128-element block of the thread's row
// into the FP8 main gradient: g = decode(code) * m_old + y (FP32: one
// rounded multiply, then one rounded add), then the block is requantised
// (m_new = max|g| / 448, codes E4M3(g * 448 / max|g|)).  `old` holds the
// block's 128 current codes; the new codes go to the staging row at `orow`
// (swizzled).  load32 and y_row as for compress_block.
template <class Load>
__device__ __forceinline__ void agoq_block(Load &&load32, float *y_row, const uint8_t *old, float m_old, uint32_t orow,
                                           uint32_t swz, float &m_new)
{
    float2 g[64];
    const float2 m2 = make_float2(m_old, m_old);
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        uint4 q;
        asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
                     : "l"(old + 16 * h));
        decode16_f2(q, g + 8 * h);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            g[8 * h + i] = mul2_rounded(g[8 * h + i], m2);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float x[32];
        load32(j, x);
        if (y_row) {
            float4 *yo = reinterpret_cast<float4 *>(y_row + 32 * j);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                yo[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
        }
#pragma unroll
        for (int t = 0; t < 16; ++t)
            g[16 * j + t] = add2_rounded(g[16 * j + t], make_float2(x[2 * t], x[2 * t + 1]));
    }
    float q;
    agoq_scales(lane_max_abs<64>(g), q, m_new);
    uint4 oq[8];
    encode_codes<64>(g, q, oq);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        sts128(orow + ((static_cast<uint32_t>(j) << 4) ^ swz), oq[j].x, oq[j].y, oq[j].z, oq[j].w);
}

// The epilogues.  kEpiCompress: the TACO compressor (codes, alpha and s
// out).  kEpiAgoq: the AGoQ accumulation into the FP8 main gradient (codes
// and the multipliers in `scale_out` read and rewritten in place).  4, 5, 6
// or 8: AGoQ's LAAQ activation quantisation at that many bits (packed codes
// and multipliers out).
constexpr int kEpiCompress = 0, kEpiAgoq = 1;
__host__ __device__ constexpr bool epi_is_laaq(int epi) { return epi >= 4; }
// Bytes of one 128-element block's output in a row of the staging tile.
__host__ __device__ constexpr int epi_block_bytes(int epi) { return epi_is_laaq(epi) ? 16 * epi : 128; }

// AGoQ 2.A quantisation (the GEMM-fused form of 2.C) of one 128-element
// block of the thread's row: amax = max|y|, q = qmax / amax, codes
// rint(y q) (the clamp to +-qmax never binds), m = amax / qmax, all in fp32
// as the stand-alone quantizer computes them.  The 128 codes, BITS bits
// each in a little-endian stream, go to the staging row at `orow` (16 BITS
// bytes, unswizzled); load32 and y_row as for compress_block.
template <int BITS, class Load>
__device__ __forceinline__ void laaq_block(Load &&load32, float *y_row, uint32_t orow, float &m)
{
    float v[128];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float x[32];
        load32(j, x);
        if (y_row) {
            float4 *yo = reinterpret_cast<float4 *>(y_row + 32 * j);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                yo[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v[32 * j + i] = x[i];
            amax = fmaxf(amax, fabsf(x[i]));
        }
    }
    float q;
    laaq_factors<BITS>(amax, q, m);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t c[32], w[BITS];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            c[i] = __float_as_uint(__fadd_rn(__fmul_rn(v[32 * j + i], q), kRoundMagic));
        pack32<BITS>(c, w);
        // 32 codes = BITS words at byte 4 BITS j of the row: 16-byte aligned
        // at 4 and 8 bits, 8-byte at 6, 4-byte at 5
        const uint32_t at = orow + 4 * BITS * j;
        if constexpr (BITS % 4 == 0) {
#pragma unroll
            for (int k = 0; k < BITS; k += 4)
                sts128(at + 4 * k, w[k], w[k + 1], w[k + 2], w[k + 3]);
        } else if constexpr (BITS % 2 == 0) {
#pragma unroll
            for (int k = 0; k < BITS; k += 2)
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(at + 4 * k), "r"(w[k]), "r"(w[k + 1]) : "memory");
        } else {
#pragma unroll
            for (int k = 0; k < BITS; ++k)
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(at + 4 * k), "r"(w[k]) : "memory");
        }
    }
}

// The last piece's warp of a split tile: for its row, the sum over the
// pieces p = 0 .. S-1 of the partials, added in that order, its own piece
// (`own`) taken from the accumulator at `tq` and the others from the
// workspace (`parts`: piece 0's [column / 4][row][4] array, offset to the
// row); the sum goes back into the accumulator.  CH chunks of 32 columns
// at a time, the other pieces' loads for them all issued before the first
// add (the loop is bound by the latency of L2).
template <int S, int BN, int CH>
__device__ __forceinline__ void sum_pieces(const float4 *parts, int own, uint32_t tq)
{
#pragma unroll 1
    for (int j0 = 0; j0 < BN / 32; j0 += CH) {
        float4 o[S - 1][CH][8];
#pragma unroll
        for (int p = 0; p < S - 1; ++p) {
            const float4 *src = parts + static_cast<int64_t>(p < own ? p : p + 1) * (kBM * BN / 4) + 8 * j0 * kBM;
#pragma unroll
            for (int c = 0; c < CH; ++c)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    o[p][c][k] = __ldcg(src + (8 * c + k) * kBM);
        }
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            float x[32];
            tmem_load_32(tq + 32 * (j0 + c), x);
            float acc[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                // piece 0
                const float4 v0 = own == 0 ? make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]) : o[0][c][k];
                acc[4 * k] = v0.x;
                acc[4 * k + 1] = v0.y;
                acc[4 * k + 2] = v0.z;
                acc[4 * k + 3] = v0.w;
            }
#pragma unroll
            for (int p = 1; p < S; ++p) {
                const int lo = p < S - 1 ? p : S - 2;  // (a constant once unrolled)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    // piece p is o[p] below the own piece, o[p - 1] above it
                    const float4 v = p == own ? make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3])
                                              : (p < own ? o[lo][c][k] : o[p - 1][c][k]);
                    acc[4 * k] = __fadd_rn(acc[4 * k], v.x);
                    acc[4 * k + 1] = __fadd_rn(acc[4 * k + 1], v.y);
                    acc[4 * k + 2] = __fadd_rn(acc[4 * k + 2], v.z);
                    acc[4 * k + 3] = __fadd_rn(acc[4 * k + 3], v.w);
                }
            }
            tmem_store_32(tq + 32 * (j0 + c), acc);
        }
    }
}

// The CTA's work: item i is global index blockIdx.x + i * gridDim.x.  The
// first `full_tiles` indices are whole tiles; the rest are pieces of the
// remaining tiles, each split along K into `split` pieces of equal length
// (the split tail: it spreads the partial last round of tiles over every
// SM).  Returns false past the end.
struct WorkItem {
    int m0, n0, kb0, kb1;
    int tail;  // the split tile's index among the tail tiles, or -1 for a whole tile
    int part;
};

__device__ __forceinline__ bool work_item(int idx, int full_tiles, int ntiles, int split, int ntn, int BN, int KB,
                                          WorkItem &w)
{
    int t;
    if (idx < full_tiles) {
        t = idx;
        w.kb0 = 0;
        w.kb1 = KB;
        w.tail = -1;
        w.part = 0;
    } else {
        const int u = idx - full_tiles;
        if (u >= (ntiles - full_tiles) * split)
            return false;
        w.tail = u / split;
        w.part = u - w.tail * split;
        t = full_tiles + w.tail;
        const int per = KB / split;
        w.kb0 = w.part * per;
        w.kb1 = w.kb0 + per;
    }
    w.m0 = (t / ntn) * kBM;
    w.n0 = (t % ntn) * BN;
    return true;
}

// EPI selects the epilogue (kEpiCompress, kEpiAgoq, or LAAQ bits; alpha_out
// is written by the compressor only, old_codes read by the AGoQ
// accumulation only; c_map is the codes' or packed codes' tensor map).
// Split-tail pieces write their fp32 partial tile to
// `ws_partial`; for each quarter of a split tile's rows, the epilogue warp
// that completes the last piece (counted in `ws_count`, 4 counters per tail
// tile, which it resets to 0) sums the pieces in piece order and runs the
// epilogue on the sum, so the result does not depend on which piece ends
// last.  No warp waits for another CTA.
template <int BN, int EPI>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_epilogue_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap b_map,
                         const __grid_constant__ CUtensorMap c_map, const uint8_t *__restrict__ old_codes,
                         float *__restrict__ alpha_out, float *__restrict__ scale_out, float *__restrict__ y_out,
                         float *__restrict__ ws_partial, unsigned int *__restrict__ ws_count, int64_t N, int K,
                         int ntiles, int full_tiles, int split, float e_target, float eps)
{
    using C = GemmCfg<BN>;
    constexpr int kGStages = C::kStages;
    constexpr uint32_t kGStageBytes = C::kStageBytes, kAccCols = C::kAccCols, kTmemCols = C::kTmemCols;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t stage_out = base + kGStages * kGStageBytes;
    const uint32_t bars = stage_out + C::kStageOut;
    const uint32_t tmem_slot = bars + C::kBars;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = K / kBK;
    const int ntn = static_cast<int>(N / BN);  // tiles along N
    const int G = gridDim.x;
    auto full = [&](int s) { return bars + 8 * s; };
    auto empty = [&](int s) { return bars + 8 * (kGStages + s); };
    auto acc_full = [&](int a) { return bars + 8 * (2 * kGStages + a); };
    auto acc_empty = [&](int a) { return bars + 8 * (2 * kGStages + 2 + a); };
    auto stage_a = [&](int s) { return base + s * kGStageBytes; };
    auto stage_b = [&](int s) { return base + s * kGStageBytes + kABytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);   // one tcgen05.commit
            mbar_init(acc_empty(a), 4);  // one arrival per epilogue warp
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    pdl_wait();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = lds32(tmem_slot);

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_map(&a_map);
            tma_prefetch_map(&b_map);
            int g = 0;  // k-blocks issued so far (all items): stage g % S, phase (g / S) & 1
            bool ok = true;
            WorkItem w;
            for (int idx = blockIdx.x; ok && work_item(idx, full_tiles, ntiles, split, ntn, BN, KB, w); idx += G) {
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                    const int s = g % kGStages;
                    if (!mbar_wait(empty(s), ((g / kGStages) & 1) ^ 1)) {
                        atomicOr(&g_gemm_error, kErrGemm);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full(s), kGStageBytes);
                    tma_load_2d(stage_a(s), &a_map, kb * kBK, w.m0, full(s));
                    tma_load_2d(stage_b(s), &b_map, kb * kBK, w.n0, full(s));
                }
            }
            // leave no load in flight into this CTA's shared memory
            for (int i = g > kGStages ? g - kGStages : 0; i < g; ++i)
                mbar_wait(full(i % kGStages), (i / kGStages) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32<kBM, BN>();
            int g = 0, i = 0;  // k-blocks consumed, items done
            bool ok = true;
            WorkItem w;
            for (int idx = blockIdx.x; ok && work_item(idx, full_tiles, ntiles, split, ntn, BN, KB, w);
                 idx += G, ++i) {
                const int a = i & 1;
                // the epilogue has emptied this accumulator (item i - 2)
                if (!mbar_wait(acc_empty(a), ((i >> 1) & 1) ^ 1)) {
                    atomicOr(&g_gemm_error, kErrGemm);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + a * kAccCols;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                    const int s = g % kGStages;
                    if (!mbar_wait(full(s), (g / kGStages) & 1)) {
                        atomicOr(&g_gemm_error, kErrGemm);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t ad = smem_desc_k_sw128(stage_a(s)), bd = smem_desc_k_sw128(stage_b(s));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)  // 16 elements = 32 bytes = 2 descriptor units
                        mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb > w.kb0) || k != 0);
                    mma_commit(empty(s));  // the stage is free once these MMAs have read it
                }
                mma_commit(acc_full(a));  // the accumulator is complete once every MMA has
            }
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const uint32_t outw = stage_out + q * C::kBlocks * 4096;  // this warp's staging tiles
        const uint32_t swz = static_cast<uint32_t>(lane & 7) << 4;
        const int64_t nblk_row = N / 128;
        int i = 0;
        WorkItem w;
        for (int idx = blockIdx.x; work_item(idx, full_tiles, ntiles, split, ntn, BN, KB, w); idx += G, ++i) {
            const int a = i & 1;
            const int m0 = w.m0, n0 = w.n0;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(acc_full(a), (i >> 1) & 1))) {
                if (lane == 0)
                    atomicOr(&g_gemm_error, kErrGemm);
                break;
            }
            tc_fence_after_sync();
            const uint32_t tq = tmem + a * kAccCols + (static_cast<uint32_t>(32 * q) << 16);
            if (w.tail >= 0) {
                // a piece of a split tile: this warp's 32 rows of fp32
                // partials to the workspace, laid out [column / 4][row][4]
                // so that a warp's 16-byte stores form one 512-byte run
                float4 *part = reinterpret_cast<float4 *>(ws_partial) +
                               (static_cast<int64_t>(w.tail) * split + w.part) * (kBM * BN / 4) + row;
#pragma unroll 1
                for (int j = 0; j < BN / 32; ++j) {
                    float x[32];
                    tmem_load_32(tq + 32 * j, x);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        __stcg(part + (8 * j + k) * kBM, make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]));
                }
                // count this warp's rows in; the warp that brings the count
                // of rows 32 q .. 32 q + 31 to `split` finishes them
                __threadfence();
                __syncwarp();
                uint32_t last = 0;
                if (lane == 0) {
                    unsigned int *cnt = ws_count + 4 * w.tail + q;
                    last = atomicAdd(cnt, 1u) == static_cast<unsigned int>(split - 1);
                    if (last)
                        *cnt = 0;  // ready for the next call
                }
                if (!__shfl_sync(0xFFFFFFFFu, last, 0)) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(acc_empty(a));
                    continue;
                }
                __threadfence();
                // the sum of the pieces, in piece order, into this
                // accumulator (which holds this CTA's own piece)
                const float4 *parts = reinterpret_cast<const float4 *>(ws_partial) +
                                      static_cast<int64_t>(w.tail) * split * (kBM * BN / 4) + row;
                switch (split) {
                case 2: sum_pieces<2, BN, 2>(parts, w.part, tq); break;
                case 3: sum_pieces<3, BN, 1>(parts, w.part, tq); break;
                default: sum_pieces<4, BN, 1>(parts, w.part, tq); break;
                }
            }
            if (lane == 0)
                bulk_wait_read_all();  // the previous tile's stores have read the staging tiles
            __syncwarp();
            float *yrow = y_out ? y_out + (m0 + row) * N + n0 : nullptr;
            const int64_t bi = static_cast<int64_t>(m0 + row) * nblk_row + n0 / 128;
            float al[C::kBlocks], sc[C::kBlocks];
#pragma unroll
            for (int blk = 0; blk < C::kBlocks; ++blk) {
                float *yb = yrow ? yrow + 128 * blk : nullptr;
                const uint32_t orow = outw + blk * 4096 + lane * epi_block_bytes(EPI);
                const uint32_t tb = tq + 128 * blk;
                auto load32 = [&](int j, float (&x)[32]) { tmem_load_32(tb + 32 * j, x); };
                if constexpr (EPI == kEpiAgoq)
                    agoq_block(load32, yb, old_codes + (m0 + row) * N + n0 + 128 * blk, scale_out[bi + blk], orow,
                               swz, sc[blk]);
                else if constexpr (EPI == kEpiCompress)
                    compress_block(load32, yb, orow, swz, e_target, eps, al[blk], sc[blk]);
                else
                    laaq_block<EPI>(load32, yb, orow, sc[blk]);
            }
            // every tensor-memory read of this accumulator is done: hand it back
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acc_empty(a));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                for (int blk = 0; blk < C::kBlocks; ++blk)  // x in bytes: a multiple of 16
                    tma_store_2d(&c_map, (n0 + blk * 128) / 128 * epi_block_bytes(EPI), m0 + 32 * q,
                                 outw + blk * 4096);
                bulk_commit();
            }
#pragma unroll
            for (int blk = 0; blk < C::kBlocks; ++blk) {
                if constexpr (EPI == kEpiCompress)
                    alpha_out[bi + blk] = al[blk];
                scale_out[bi + blk] = sc[blk];
            }
        }
        if (lane == 0)
            bulk_wait_all();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

constexpr int kMaxDevices = 64;

}  // namespace

cudaError_t read_gemm_error(uint32_t *flags, bool clear)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof v);
    if (e != cudaSuccess)
        return e;
    *flags = v;
    if (clear) {
        v = 0;
        e = cudaMemcpyToSymbol(g_gemm_error, &v, sizeof v);
    }
    return e;
}

namespace {

// The split tail.  A persistent grid of G CTAs (one per SM) takes the
// tiles in rounds of G; when the tile count T is not a multiple of G, the
// last round leaves SMs idle.  Instead, the rem = T mod G tiles of that round
// (all T tiles when T < G) are each cut along K into S pieces, and the
// rem * S pieces are dealt out like tiles; a piece costs 1/S of a tile, so
// the tail costs ceil(rem S / G) / S rounds instead of one.  S is the
// smallest of 1..4 dividing the k-block count that brings the tail's cost
// down the most, and a split is taken only if it saves at least 1/8 of a
// round (the pieces' partial sums go through L2), if each piece spans at
// least kMinPieceKB k-blocks, and if the workspace holds it.  The piece
// length bound keeps the MMAs ahead of the epilogue warps: a piece's MMAs
// must outlast the epilogue of the item before it (a tile's compression,
// or a piece's partial store and, for the last piece, the sum and the
// compression), else the MMA warp waits for a free accumulator.  Measured
// on the GPT-6.7B down-projection (8192 x 4096 x 4096, 1024 tiles): the
// split of its last 112 tiles into pieces of 16 k-blocks took 175-179 us
// against 150-157 us unsplit, the tensor pipe active 77 % of the time
// against 84 %; the weight gradient (4096 x 4096 x 8192, 512 tiles), split
// into pieces of 64 k-blocks, went from 181-185 us to 168-173 us.
constexpr int kMinPieceKB = 32;
struct TailPlan {
    int grid = 0, full_tiles = 0, split = 1, tail_tiles = 0;
    uint64_t ws_bytes = 0;  // workspace the split needs (0: no split)
};

// The workspace starts with the arrival counters, 4 per tail tile, at a
// place and of a size that do not depend on the shape (fewer tail tiles than
// SMs): every call leaves the counters it used at zero, and no call writes
// partial sums over them, so one workspace serves calls of any shape.
uint64_t count_bytes(int sms) { return (16 * static_cast<uint64_t>(sms) + 255) & ~uint64_t(255); }

TailPlan plan_tail(int64_t ntiles, int64_t KB, int BN, int sms, uint64_t ws_avail)
{
    TailPlan p;
    const int64_t rem = ntiles >= sms ? ntiles % sms : ntiles;
    double best = rem > 0 ? 1.0 : 0.0;
    for (int S = 2; S <= 4; ++S) {
        if (KB % S != 0 || KB / S < kMinPieceKB)
            continue;
        const double cost = static_cast<double>((rem * S + sms - 1) / sms) / S;
        const uint64_t ws = count_bytes(sms) + static_cast<uint64_t>(rem) * S * kBM * BN * 4;
        if (cost <= best - 0.125) {
            best = cost;
            p.split = S;
            p.ws_bytes = ws;
        }
    }
    if (p.ws_bytes > ws_avail) {  // no room for the best split: none
        p.split = 1;
        p.ws_bytes = 0;
    }
    p.tail_tiles = p.split > 1 ? static_cast<int>(rem) : 0;
    p.full_tiles = static_cast<int>(ntiles - p.tail_tiles);
    const int64_t units = p.full_tiles + static_cast<int64_t>(p.tail_tiles) * p.split;
    p.grid = static_cast<int>(units < sms ? units : sms);
    return p;
}

template <int BN, int EPI>
cudaError_t run_gemm(const CUtensorMap &am, const void *b_bf16, int64_t M, int64_t N, int64_t K, float e_target,
                     float eps, uint8_t *codes, const CUtensorMap &cm, float *alpha, float *scale, float *y_out,
                     void *workspace, uint64_t workspace_bytes, const DeviceInfo &di, cudaStream_t stream)
{
    using C = GemmCfg<BN>;
    CUtensorMap bm;
    if (encode_tensor_map_2d(&bm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(b_bf16), K, N, K * 2, kBK,
                             BN) != 0)
        return cudaErrorInvalidValue;
    static std::atomic<bool> set[kMaxDevices];
    if (!set[di.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(gemm_epilogue_kernel<BN, EPI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem));
        if (e != cudaSuccess)
            return e;
        set[di.device].store(true, std::memory_order_release);
    }
    const int64_t ntiles = (M / kBM) * (N / BN);
    const TailPlan p = plan_tail(ntiles, K / kBK, BN, di.num_sms, workspace ? workspace_bytes : 0);
    unsigned int *count = p.split > 1 ? static_cast<unsigned int *>(workspace) : nullptr;
    float *partial =
        p.split > 1 ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + count_bytes(di.num_sms)) : nullptr;
    return launch_pdl(gemm_epilogue_kernel<BN, EPI>, p.grid, kGThreads, C::kSmem, stream, am, bm, cm,
                      static_cast<const uint8_t *>(codes), alpha, scale, y_out, partial, count, N,
                      static_cast<int>(K), static_cast<int>(ntiles), p.full_tiles, p.split, e_target, eps);
}

// 256-wide tiles whenever N allows, 128-wide otherwise.  With a one-CTA MMA
// a 128-wide tile does half the arithmetic per byte of A it reads from shared
// memory: measured on the GPT-6.7B shapes, 128-wide tiles took 226 us where
// 256-wide ones took 152 us (down-projection, 8192 x 4096 x 4096) and 181 us
// (weight gradient, 4096 x 4096 x 8192), though the latter's 1024 narrow
// tiles fill the last round of SMs better than its 512 wide ones.
int tile_width(int64_t N) { return N % 256 == 0 ? 256 : 128; }

// The codes' tensor map: one byte a code ([M][N], 128-byte rows of a
// block, swizzled like the staging rows), or LAAQ's packed stream ([M][N
// bits / 8], 16 bits bytes a block, unswizzled staging rows).
template <int EPI>
cudaError_t launch_gemm_epilogue(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                 float e_target, float eps, uint8_t *codes, float *alpha, float *scale, float *y_out,
                                 void *workspace, uint64_t workspace_bytes, cudaStream_t stream)
{
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess)
        return e;
    CUtensorMap am, cm;
    const uint64_t row_bytes = static_cast<uint64_t>(N) / 128 * epi_block_bytes(EPI);
    if (encode_tensor_map_2d(&am, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(a_bf16), K, M, K * 2, kBK,
                             kBM) != 0 ||
        encode_tensor_map_2d(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, row_bytes, M, row_bytes,
                             epi_block_bytes(EPI), 32,
                             epi_is_laaq(EPI) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B) != 0)
        return cudaErrorInvalidValue;
    if (tile_width(N) == 256)
        return run_gemm<256, EPI>(am, b_bf16, M, N, K, e_target, eps, codes, cm, alpha, scale, y_out, workspace,
                                  workspace_bytes, di, stream);
    return run_gemm<128, EPI>(am, b_bf16, M, N, K, e_target, eps, codes, cm, alpha, scale, y_out, workspace,
                              workspace_bytes, di, stream);
}

}  // namespace

cudaError_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, uint64_t *bytes)
{
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess)
        return e;
    const int BN = tile_width(N);
    *bytes = plan_tail((M / kBM) * (N / BN), K / kBK, BN, di.num_sms, ~uint64_t(0)).ws_bytes;
    return cudaSuccess;
}

cudaError_t launch_gemm_compress(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                 float e_target, float eps, uint8_t *codes, float *alpha, float *scale,
                                 float *y_out, void *workspace, uint64_t workspace_bytes, cudaStream_t stream)
{
    return launch_gemm_epilogue<kEpiCompress>(a_bf16, b_bf16, M, N, K, e_target, eps, codes, alpha, scale, y_out,
                                              workspace, workspace_bytes, stream);
}

cudaError_t launch_gemm_agoq_accumulate(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                        uint8_t *main_codes, float *main_scale, float *y_out, void *workspace,
                                        uint64_t workspace_bytes, cudaStream_t stream)
{
    return launch_gemm_epilogue<kEpiAgoq>(a_bf16, b_bf16, M, N, K, 1.0f, 1.0f, main_codes, nullptr, main_scale,
                                          y_out, workspace, workspace_bytes, stream);
}

cudaError_t launch_gemm_laaq_quantize(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                      int bits, uint8_t *packed, float *scale, float *y_out, void *workspace,
                                      uint64_t workspace_bytes, cudaStream_t stream)
{
    switch (bits) {
    case 4:
        return launch_gemm_epilogue<4>(a_bf16, b_bf16, M, N, K, 1.0f, 1.0f, packed, nullptr, scale, y_out, workspace,
                                       workspace_bytes, stream);
    case 5:
        return launch_gemm_epilogue<5>(a_bf16, b_bf16, M, N, K, 1.0f, 1.0f, packed, nullptr, scale, y_out, workspace,
                                       workspace_bytes, stream);
    case 6:
        return launch_gemm_epilogue<6>(a_bf16, b_bf16, M, N, K, 1.0f, 1.0f, packed, nullptr, scale, y_out, workspace,
                                       workspace_bytes, stream);
    case 8:
        return launch_gemm_epilogue<8>(a_bf16, b_bf16, M, N, K, 1.0f, 1.0f, packed, nullptr, scale, y_out, workspace,
                                       workspace_bytes, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace taco
