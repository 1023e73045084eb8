// Fused shard reduce + decompress for sm_103a: the reducing rank of the
// two-shot AllReduce (TACO, gist.science summary of arXiv 2604.24088, 2.B.3)
// both sends the compressed reduced shard (AllGather payload) and uses its
// reconstruction.  One pass writes the compressed sum (codes, alpha, s) and
// decompress(compressed sum) without reading the reduced codes back.
//
// The one-pass kernel is for n=128 (taco_reduce_decompress128_kernel
// below).  For n=256 the call runs the shard-reduce kernel and then the
// decompress kernel: a one-pass n=256 kernel (32-row tiles, one CTA per SM)
// took 135.5 us per call at P=8 x [8192, 5120] against 116.4 us for the two
// launches, because its row-resident phase 2 and the P shards' loads leave
// room for only one CTA (8 warps) per SM.

#include <atomic>
#include <cfloat>

#include "codec_math.cuh"
#include "device_utils.cuh"
#include "internal.h"
#include "reduce_math.cuh"

namespace taco {

namespace {

constexpr int kFWarps = 8;
constexpr int kFThreads = kFWarps * 32;

// ------------------------------------------------- n = 128, two CTAs/SM --
//
// Each warp takes 16-row tiles (16 blocks), laid out so that two CTAs fit
// per SM (at most 128 registers a thread):
//  phase 1  16 elements per lane (8 lanes per block, 4 blocks per sub-step,
//           4 sub-steps per 16-row tile), the next sub-step's shard loads in
//           flight for P <= 8; block statistics in the canonical order, so
//           codes and scalars equal the shard-reduce kernel's.
//  phase 2  lane pairs: lane 2r + h decompresses elements 64h .. 64h + 63 of
//           tile row r, with the decompress kernel's arithmetic operation for
//           operation (the last butterfly stage takes the partner's values by
//           shuffle), so the output equals taco_decompress's.
constexpr int kPRows = 16;                                   // tile rows (= blocks)
constexpr uint32_t kPCodeTile = kPRows * 128;                // 2 KB
constexpr uint32_t kPOutBytes = kPRows * 512;                // 8 KB
constexpr uint32_t kPWarpBytes = kPCodeTile + kPOutBytes;    // 10 KB
constexpr uint32_t kPScalarBytes = 2 * kPRows * 4;
constexpr uint32_t kPSmemBytes = 1024 + kFWarps * (kPWarpBytes + kPScalarBytes);
static_assert(kPCodeTile % 1024 == 0 && kPOutBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");

struct Slot16 {
    int64_t blk, off;
    int lb;
    bool valid;
};

__device__ __forceinline__ Slot16 slot16(int64_t blk0, int si, int lane, int64_t nblocks)
{
    Slot16 s;
    s.lb = si * 4 + lane / 8;
    s.blk = blk0 + s.lb;
    s.valid = s.blk < nblocks;
    s.off = (s.valid ? s.blk : 0) * 128 + (lane % 8) * 16;
    return s;
}

template <int P>
__device__ __forceinline__ void load_shards16(const ShardPtrs &in, const Slot16 &sl, uint64_t pol, uint4 (&q)[P][1])
{
#pragma unroll
    for (int p = 0; p < P; ++p)
        q[p][0] = sl.valid ? ldg128_stream_hint(in.codes[p] + sl.off, pol) : make_uint4(0, 0, 0, 0);
}

// T = sum_p decode(q_p) w_p for a compile-time shard count (weights loaded
// by lane `part` for shards part, part + 8, ... and broadcast).
template <int P>
__device__ __forceinline__ void accumulate16_fixed(const ShardPtrs &in, const Slot16 &sl, const uint4 (&q)[P][1],
                                                   int lane, float2 (&T)[8])
{
    constexpr int ROUNDS = (P + 7) / 8;
    const int part = lane % 8;
    float wr[ROUNDS];
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const int p = r * 8 + part;
        const bool ok = sl.valid && p < P;
        wr[r] = shard_weight(ok ? __ldg(in.scale[p] + sl.blk) : 1.0f, ok ? __ldg(in.alpha[p] + sl.blk) : 1.0f);
    }
    const int gbase = lane & ~7;
    float w[P];
#pragma unroll
    for (int p = 0; p < P; ++p)
        w[p] = __shfl_sync(0xFFFFFFFFu, wr[p / 8], gbase + (p % 8));
    weighted_sum<P, 8>(q, w, T);
}

__device__ __forceinline__ void accumulate16_any(const ShardPtrs &in, int P, const Slot16 &sl, uint64_t pol,
                                                 float2 (&T)[8])
{
#pragma unroll 1
    for (int p = 0; p < P; ++p) {
        uint4 q[1];
        load_codes<8, true>(in.codes[p] + sl.off, sl.valid, q, pol);
        const float w = sl.valid ? shard_weight(__ldg(in.scale[p] + sl.blk), __ldg(in.alpha[p] + sl.blk)) : 1.0f;
        weighted_sum_step<8>(q, w, p == 0, T);
    }
}

// Requantises the lane's 16 sums, stores its code word and (lane part 0)
// the block scalars to global memory and to the warp's shared tile.
__device__ __forceinline__ void finish16(float2 (&T)[8], const Slot16 &sl, int lane, float e_target, float eps,
                                         uint8_t *out_codes, float *out_alpha, float *out_scale, uint32_t ctile,
                                         float *sa_s, float *ss_s)
{
    const int part = lane % 8;
    uint4 oq[1];
    float alpha, scale;
    recompress<128, 8, 8>(T, e_target, eps, oq, alpha, scale);
    if (sl.valid) {
        stg128_stream(out_codes + sl.off, oq[0]);
        if (part == 0) {
            out_alpha[sl.blk] = alpha;
            out_scale[sl.blk] = scale;
        }
    }
    const int r = sl.lb;
    const uint32_t rsw = static_cast<uint32_t>(r & 7) << 4;
    sts128(ctile + r * 128 + ((static_cast<uint32_t>(part) << 4) ^ rsw), oq[0].x, oq[0].y, oq[0].z, oq[0].w);
    if (part == 0) {
        sa_s[sl.lb] = alpha;
        ss_s[sl.lb] = scale;
    }
}

// Stages h = 2 .. 32 (element strides) of the transform on a half row of 64
// elements held as 32 float2: the in-lane stages of the lane-pair layout.
__device__ __forceinline__ void fwht64_upper(float2 (&v)[32])
{
#pragma unroll
    for (int hh = 1; hh < 32; hh <<= 1) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if ((k & hh) == 0) {
                const float2 a = v[k], b = v[k + hh];
                v[k] = __fadd2_rn(a, b);
                v[k + hh] = sub2(a, b);
            }
        }
    }
}

template <int PT, bool BF16OUT>
__global__ void __launch_bounds__(kFThreads, 2)
    taco_reduce_decompress128_kernel(const ShardPtrs in, int P, const __grid_constant__ CUtensorMap o_map,
                                     int64_t nrows, float e_target, float eps, uint8_t *__restrict__ out_codes,
                                     float *__restrict__ out_alpha, float *__restrict__ out_scale)
{
    constexpr int SUB = 4;  // phase-1 sub-steps per 16-row tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t outw = base + warp * kPOutBytes;                         // 8 KB, 1 KB aligned
    const uint32_t ctile = base + kFWarps * kPOutBytes + warp * kPCodeTile;  // 2 KB, 1 KB aligned
    float *sa_s = reinterpret_cast<float *>(smem_raw + (base - raw) + kFWarps * kPWarpBytes + warp * kPScalarBytes);
    float *ss_s = sa_s + kPRows;

    pdl_wait();
    pdl_launch_dependents();
    if (lane == 0)
        tma_prefetch_map(&o_map);
    const int64_t nblocks = nrows;
    const int64_t ntiles = (nrows + kPRows - 1) / kPRows;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kFWarps + warp;
    const int64_t W = static_cast<int64_t>(gridDim.x) * kFWarps;
    const int r = lane >> 1, h = lane & 1;
    const uint32_t swz = static_cast<uint32_t>(r & 7) << 4;
    // evict-first L2 policy: the shards' codes and the output are touched once
    const uint64_t pol = policy_evict_first();

    for (int64_t t = gw; t < ntiles; t += W) {
        const int64_t blk0 = t * kPRows;
        // ------------------------------------------------------ phase 1
        if constexpr (PT > 0) {
            uint4 qa[PT][1], qb[PT][1];
            Slot16 sa = slot16(blk0, 0, lane, nblocks), sb;
            load_shards16<PT>(in, sa, pol, qa);
#pragma unroll
            for (int si = 0; si < SUB; si += 2) {
                sb = slot16(blk0, si + 1, lane, nblocks);
                load_shards16<PT>(in, sb, pol, qb);
                float2 T[8];
                accumulate16_fixed<PT>(in, sa, qa, lane, T);
                finish16(T, sa, lane, e_target, eps, out_codes, out_alpha, out_scale, ctile, sa_s, ss_s);
                if (si + 2 < SUB) {
                    sa = slot16(blk0, si + 2, lane, nblocks);
                    load_shards16<PT>(in, sa, pol, qa);
                }
                accumulate16_fixed<PT>(in, sb, qb, lane, T);
                finish16(T, sb, lane, e_target, eps, out_codes, out_alpha, out_scale, ctile, sa_s, ss_s);
            }
        } else {
#pragma unroll 1
            for (int si = 0; si < SUB; ++si) {
                const Slot16 sl = slot16(blk0, si, lane, nblocks);
                float2 T[8];
                accumulate16_any(in, P, sl, pol, T);
                finish16(T, sl, lane, e_target, eps, out_codes, out_alpha, out_scale, ctile, sa_s, ss_s);
            }
        }
        __syncwarp();

        // ------------------------------------------------------ phase 2
        const float a = sa_s[r], sc = ss_s[r];
        float2 w64[64];  // decode helpers index a 64-entry row; this lane fills entries 0 .. 31
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            decode16_stage1(lds128(ctile + r * 128 + ((static_cast<uint32_t>(4 * h + jj) << 4) ^ swz)), w64, jj);
        float2 v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k)
            v[k] = w64[k];
        fwht64_upper(v);
        // the multiplier as in decompress_multiplier, then the last stage
        // fused with it as in last_stage_scaled, across the lane pair
        const float c = BlockConst<128>::c;
        const float sa2 = sc * a;
        float kk = c / sa2;
        if (!(sa2 <= FLT_MAX) || !(kk >= FLT_MIN)) {
            const float inv_s = 1.0f / sc;
            const float2 i2 = make_float2(inv_s, inv_s);
#pragma unroll
            for (int k = 0; k < 32; ++k)
                v[k] = __fmul2_rn(v[k], i2);
            kk = c / a;
        }
        const float2 k2 = make_float2(kk, kk), nk2 = make_float2(-kk, -kk);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            float2 o;
            o.x = __shfl_xor_sync(0xFFFFFFFFu, v[k].x, 1);
            o.y = __shfl_xor_sync(0xFFFFFFFFu, v[k].y, 1);
            const float2 av = h ? o : v[k], bv = h ? v[k] : o;  // elements i and i + 64
            const float2 ak = __fmul2_rn(av, k2);
            v[k] = __ffma2_rn(bv, h ? nk2 : k2, ak);
        }
        if (lane == 0)
            bulk_wait_read_all();
        __syncwarp();
        if constexpr (!BF16OUT) {
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                const uint32_t b = 2 * h + (ch >> 3), j = ch & 7;
                sts128(outw + b * 2048 + r * 128 + ((j << 4) ^ swz), __float_as_uint(v[2 * ch].x),
                       __float_as_uint(v[2 * ch].y), __float_as_uint(v[2 * ch + 1].x), __float_as_uint(v[2 * ch + 1].y));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                sts128(outw + h * 2048 + r * 128 + ((static_cast<uint32_t>(j) << 4) ^ swz),
                       f32x2_to_bf16x2(v[4 * j].x, v[4 * j].y), f32x2_to_bf16x2(v[4 * j + 1].x, v[4 * j + 1].y),
                       f32x2_to_bf16x2(v[4 * j + 2].x, v[4 * j + 2].y), f32x2_to_bf16x2(v[4 * j + 3].x, v[4 * j + 3].y));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            constexpr int nbox = BF16OUT ? 2 : 4;
            constexpr int box_inner = BF16OUT ? 64 : 32;
            // the output is written once and not read again here: same policy
#pragma unroll
            for (int b = 0; b < nbox; ++b)
                tma_store_2d_hint(&o_map, b * box_inner, static_cast<int32_t>(t * kPRows), outw + b * 2048, pol);
            bulk_commit();
        }
        __syncwarp();  // the code tile and scalars are rewritten by the next tile's phase 1
    }
    if (lane == 0)
        bulk_wait_all();
}

template <int PT, bool BF> std::atomic<bool> g_smem128_set[64];

template <int PT, bool BF>
cudaError_t run_fused128(const ShardPtrs &in, int P, const CUtensorMap &om, int64_t nrows, float e_target,
                         float eps, uint8_t *oc, float *oa, float *os, cudaStream_t st, const DeviceInfo &di)
{
    auto kernel = taco_reduce_decompress128_kernel<PT, BF>;
    if (!g_smem128_set<PT, BF>[di.device].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kPSmemBytes));
        if (e != cudaSuccess)
            return e;
        g_smem128_set<PT, BF>[di.device].store(true, std::memory_order_release);
    }
    const int64_t ctas = (nrows + kFWarps * kPRows - 1) / (kFWarps * kPRows);
    const int grid = static_cast<int>(ctas < 2 * di.num_sms ? ctas : 2 * di.num_sms);
    return launch_pdl(kernel, grid, kFThreads, kPSmemBytes, st, in, P, om, nrows, e_target, eps, oc, oa, os);
}

template <bool BF>
cudaError_t dispatch_p128(const ShardPtrs &in, int P, const CUtensorMap &om, int64_t nrows, float e_target,
                          float eps, uint8_t *oc, float *oa, float *os, cudaStream_t st, const DeviceInfo &di)
{
    switch (P) {
    case 2:
        return run_fused128<2, BF>(in, P, om, nrows, e_target, eps, oc, oa, os, st, di);
    case 4:
        return run_fused128<4, BF>(in, P, om, nrows, e_target, eps, oc, oa, os, st, di);
    case 8:
        return run_fused128<8, BF>(in, P, om, nrows, e_target, eps, oc, oa, os, st, di);
    default:
        return run_fused128<0, BF>(in, P, om, nrows, e_target, eps, oc, oa, os, st, di);
    }
}

}  // namespace

cudaError_t launch_reduce_decompress(int P, const ShardPtrs &in, int64_t nrows, int block, float e_target,
                                     float eps, uint8_t *out_codes, float *out_alpha, float *out_scale,
                                     void *out, bool out_bf16, cudaStream_t stream)
{
    if (block != 128) {
        const cudaError_t e = launch_taco_reduce(P, in, nrows * 128 / block, block, e_target, eps, out_codes,
                                                 out_alpha, out_scale, stream);
        if (e != cudaSuccess)
            return e;
        return launch_decompress(out_codes, out_alpha, out_scale, nrows, block, out, out_bf16, false, stream);
    }
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess)
        return e;
    CUtensorMap om;
    const int rc = out_bf16
                       ? encode_tensor_map_2d(&om, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, 128, nrows, 256, 64, kPRows)
                       : encode_tensor_map_2d(&om, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out, 128, nrows, 512, 32, kPRows);
    if (rc != 0)
        return cudaErrorInvalidValue;
    return out_bf16 ? dispatch_p128<true>(in, P, om, nrows, e_target, eps, out_codes, out_alpha, out_scale, stream,
                                          di)
                    : dispatch_p128<false>(in, P, om, nrows, e_target, eps, out_codes, out_alpha, out_scale,
                                           stream, di);
}

}  // namespace taco
