// Shard reduce (TACO two-shot local step) and AGoQ FP8 gradient kernels for
// sm_103a.  None of these needs a Hadamard rotation on its path, so they
// use plain coalesced 16-byte loads: a lane owns 32 (AGoQ accumulate, shard
// reduces of up to four shards) or 16 (shard reduces of more shards)
// consecutive elements of a block, adjacent lanes own one block, per-block
// statistics (sum of squares, absolute maximum) are combined with
// __shfl_xor_sync, and the per-shard scalars of a block are fetched once per
// lane group and broadcast with __shfl_sync.  For up to four shards the
// shard reduces keep the next grid-stride slot's loads in flight while they
// compute the current one.
//
// TACO shard reduce, computed in the Hadamard domain.  With c = 1/sqrt(n)
// and H the Sylvester matrix (c H c H = I), shard p decompresses to
//     x_p = c H (d_p / s_p) / alpha_p,        d_p = decode(codes_p),
// so the FP32 sum of the P reconstructions is S = c H T with
//     T = sum_p d_p / (s_p alpha_p).
// Compressing S (TACO 2.B.1-2.B.2) needs mean(S^2) = |T|^2 / n (Parseval)
// and the rotation y = c H (alpha' S) = alpha' T, hence
//     alpha' = sqrt(E / (|T|^2/n + eps)),  s' = 448 / (alpha' max|T|),
//     codes' = E4M3(alpha' s' T),
// which is the literal decompress-sum-compress result without either
// rotation.  (AGoQ 2.B, step 2: the sum is taken in FP32 so that it cannot
// overflow the FP8 range.)

#include <cfloat>

#include "device_utils.cuh"
#include "internal.h"
#include "reduce_math.cuh"

namespace taco {

namespace {

constexpr int kBlockThreads = 256;

// Elements per lane of the two reduces: 32 (two 16-byte code words per
// shard) for up to four shards, 16 (one word) above that, where the P words
// in flight per slot would otherwise cost occupancy.  The block statistics
// are bit-identical in either layout (reduce_math.cuh).
template <int P> __host__ __device__ constexpr int elems_per_lane() { return P <= 4 ? 32 : 16; }

// Whether a lane keeps its next grid-stride slot's loads in flight while it
// processes the current one (two slots of registers).
template <int P> __host__ __device__ constexpr bool prefetch_next() { return P <= 4; }

template <int NB, int P> __host__ __device__ constexpr int lanes_per_block() { return NB / elems_per_lane<P>(); }

template <int NB, int P> __host__ __device__ constexpr int rounds_of()
{
    return (P + lanes_per_block<NB, P>() - 1) / lanes_per_block<NB, P>();
}

// One grid-stride slot of a lane: its block, offset, and the loads.
template <int P, int ROUNDS, int NF> struct RedSlot {
    uint4 q[P][NF / 8];
    float sc[ROUNDS];  // scale (TACO) or dequantisation multiplier (AGoQ) of shard r * LPB + part
    float al[ROUNDS];  // alpha of that shard (TACO only)
    int64_t blk, off;
    bool valid;
};

template <int NB, int P>
using SlotOf = RedSlot<P, rounds_of<NB, P>(), elems_per_lane<P>() / 2>;

// WIDE: each shard's 32 codes come with one 32-byte load (every shard's
// codes 32-byte aligned; 32 elements per lane with an L2 policy).
template <int NB, int P, bool WITH_ALPHA, bool EF, bool WIDE = false>
__device__ __forceinline__ void load_slot(const ShardPtrs &in, int64_t base, int lane, int64_t total,
                                          uint64_t pol, SlotOf<NB, P> &s)
{
    constexpr int LPB = lanes_per_block<NB, P>();
    constexpr int NF = elems_per_lane<P>() / 2;
    const int part = lane % LPB;
    const int64_t t = base + lane;
    s.valid = t < total;
    s.blk = s.valid ? static_cast<int64_t>(static_cast<uint64_t>(t) / LPB) : 0;  // t >= 0: a shift
    s.off = s.blk * NB + part * elems_per_lane<P>();
#pragma unroll
    for (int p = 0; p < P; ++p)
        load_codes<NF, EF, WIDE>(in.codes[p] + s.off, s.valid, s.q[p], pol);
#pragma unroll
    for (int r = 0; r < rounds_of<NB, P>(); ++r) {
        const int p = r * LPB + part;
        const bool ok = s.valid && p < P;
        s.sc[r] = ok ? __ldg(in.scale[p] + s.blk) : 1.0f;
        s.al[r] = (WITH_ALPHA && ok) ? __ldg(in.alpha[p] + s.blk) : 1.0f;
    }
}

// Per-shard factors for every shard of the lane's block, from the values the
// lane group loaded (lane `part` holds shards part, part + LPB, ...).
template <int LPB, int P, int ROUNDS>
__device__ __forceinline__ void share_factors(const float (&mine)[ROUNDS], int lane, float (&f)[P])
{
    const int gbase = lane & ~(LPB - 1);
#pragma unroll
    for (int p = 0; p < P; ++p)
        f[p] = __shfl_sync(0xFFFFFFFFu, mine[p / LPB], gbase + (p % LPB));
}

// Runs `process` over the lane's grid-stride slots.  For up to four shards
// the next slot's loads are issued before the current slot is processed
// (ping-pong); with more shards the second slot's registers would cost more
// occupancy than the prefetch gains.  EF: the codes are loaded with an L2
// evict-first policy.
template <int NB, int P, bool WITH_ALPHA, bool EF, bool WIDE, typename F>
__device__ __forceinline__ void for_each_slot(const ShardPtrs &in, int64_t nblocks, F &&process)
{
    constexpr int LPB = lanes_per_block<NB, P>();
    const int64_t total = nblocks * LPB;
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
    const uint64_t pol = EF ? policy_evict_first() : 0;
    SlotOf<NB, P> a, b;
    if constexpr (!prefetch_next<P>()) {
        for (; base < total; base += stride) {
            load_slot<NB, P, WITH_ALPHA, EF, WIDE>(in, base, lane, total, pol, a);
            process(a);
        }
    } else {
        load_slot<NB, P, WITH_ALPHA, EF, WIDE>(in, base, lane, total, pol, a);
        while (base < total) {
            load_slot<NB, P, WITH_ALPHA, EF, WIDE>(in, base + stride, lane, total, pol, b);
            process(a);
            base += stride;
            if (base >= total)
                break;
            load_slot<NB, P, WITH_ALPHA, EF, WIDE>(in, base + stride, lane, total, pol, a);
            process(b);
            base += stride;
        }
    }
}

// ------------------------------------------------------ TACO reduce --

template <int NB, int P, bool WIDE>
__device__ __forceinline__ void taco_reduce_body(const ShardPtrs &in, int64_t nblocks, float e_target, float eps,
                                                 uint8_t *__restrict__ out_codes, float *__restrict__ out_alpha,
                                                 float *__restrict__ out_scale)
{
    constexpr int LPB = lanes_per_block<NB, P>();
    constexpr int NF = elems_per_lane<P>() / 2;
    constexpr int ROUNDS = rounds_of<NB, P>();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    // the shards' codes are read once: evict-first keeps L2 for the reduced
    // codes, which the decompress reads next
    for_each_slot<NB, P, true, true, WIDE>(in, nblocks, [&](const SlotOf<NB, P> &s) {
        float wr[ROUNDS];
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r)
            wr[r] = shard_weight(s.sc[r], s.al[r]);
        float w[P];
        share_factors<LPB, P, ROUNDS>(wr, lane, w);
        float2 T[NF];
        weighted_sum<P, NF>(s.q, w, T);
        uint4 oq[NF / 8];
        float alpha, scale;
        recompress<NB, LPB, NF>(T, e_target, eps, oq, alpha, scale);
        if (s.valid) {
#pragma unroll
            for (int h = 0; h < NF / 8; ++h)
                stg128_stream(out_codes + s.off + 16 * h, oq[h]);
            if (lane % LPB == 0) {
                out_alpha[s.blk] = alpha;
                out_scale[s.blk] = scale;
            }
        }
    });
}

// Up to four shards: 32 elements per lane, at most 128 registers a thread,
// two CTAs per SM.  Launched alone at the GPT-6.7B size it takes 27.1 us
// against 30.1 us with 16 elements per lane.  In the back-to-back step
// (compress, reduce, decompress launched with programmatic dependent launch)
// the step took 118.9 us against 120.3 us with 16 elements.  (While every
// kernel triggered its dependents at its start, the 32-element step took
// 132.7 us: device_utils.cuh.)  Three CTAs per SM (80 registers) measured
// 2 % slower with 16 elements.
template <int NB, int P, bool WIDE>
__global__ void __launch_bounds__(kBlockThreads, 2)
    taco_reduce_kernel(const ShardPtrs in, int64_t nblocks, float e_target, float eps,
                       uint8_t *__restrict__ out_codes, float *__restrict__ out_alpha,
                       float *__restrict__ out_scale)
{
    taco_reduce_body<NB, P, WIDE>(in, nblocks, e_target, eps, out_codes, out_alpha, out_scale);
}

// Five or more shards: the compiler's register choice (a two-CTA bound
// measured 22 % slower at P = 8).
template <int NB, int P>
__global__ void __launch_bounds__(kBlockThreads)
    taco_reduce_many_kernel(const ShardPtrs in, int64_t nblocks, float e_target, float eps,
                            uint8_t *__restrict__ out_codes, float *__restrict__ out_alpha,
                            float *__restrict__ out_scale)
{
    taco_reduce_body<NB, P, false>(in, nblocks, e_target, eps, out_codes, out_alpha, out_scale);
}

// ----------------------------------------------------- AGoQ reduce --

template <int NB, int P>
__global__ void __launch_bounds__(kBlockThreads)
    agoq_reduce_kernel(const ShardPtrs in, int64_t nblocks, uint8_t *__restrict__ out_codes,
                       float *__restrict__ out_scale)
{
    constexpr int LPB = lanes_per_block<NB, P>();
    constexpr int NF = elems_per_lane<P>() / 2;
    pdl_wait();
    const int lane = threadIdx.x & 31;
    // default L2 policy: evict-first loads measured 5% slower here
    for_each_slot<NB, P, false, false, false>(in, nblocks, [&](const SlotOf<NB, P> &s) {
        float m[P];
        share_factors<LPB, P, rounds_of<NB, P>()>(s.sc, lane, m);
        // FP32 dequantise (one rounded multiply) and FP32 sum in shard order
        float2 S[NF];
        weighted_sum<P, NF>(s.q, m, S);
        const float mx = group_max<LPB>(lane_max_abs<NF>(S));
        float qs, m_new;
        agoq_scales(mx, qs, m_new);
        uint4 oq[NF / 8];
        encode_codes<NF>(S, qs, oq);
        if (s.valid) {
#pragma unroll
            for (int h = 0; h < NF / 8; ++h)
                stg128_stream(out_codes + s.off + 16 * h, oq[h]);
            if (lane % LPB == 0)
                out_scale[s.blk] = m_new;
        }
    });
}

// ------------------------------------------------- AGoQ accumulate --

// Slots a lane takes per loop trip of the accumulate kernel; the loads of
// all of them are issued before any is processed.
constexpr int kAccSlots = 2;

template <int NB>
__global__ void __launch_bounds__(kBlockThreads)
    agoq_accumulate_kernel(uint8_t *__restrict__ codes, float *__restrict__ scale,
                           const uint16_t *__restrict__ grad, int64_t nblocks)
{
    constexpr int LPB = NB / kLaneElems;
    constexpr int U = kAccSlots;
    pdl_wait();
    const int64_t total = nblocks * LPB;
    const int lane = threadIdx.x & 31;
    const int part = lane % LPB;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
         base += U * stride) {
        uint4 q[U][2], g[U][4];
        float s_old[U];
        int64_t blk[U], off[U];
        bool valid[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t t = base + u * stride + lane;
            valid[u] = t < total;
            blk[u] = valid[u] ? t / LPB : 0;
            off[u] = blk[u] * NB + part * kLaneElems;
            s_old[u] = 1.0f;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                q[u][h] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int h = 0; h < 4; ++h)
                g[u][h] = make_uint4(0, 0, 0, 0);
            if (valid[u]) {
                // codes and scale are rewritten below: coherent loads, not .nc
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(q[u][h].x), "=r"(q[u][h].y), "=r"(q[u][h].z), "=r"(q[u][h].w)
                                 : "l"(codes + off[u] + 16 * h));
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    g[u][h] = ldg128_stream(grad + off[u] + 8 * h);
                asm volatile("ld.global.f32 %0, [%1];" : "=f"(s_old[u]) : "l"(scale + blk[u]));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            // g = dequantise(main) + grad in FP32: one rounded multiply, then
            // one rounded add (no fused multiply-add), as the stated
            // arithmetic is.
            float2 d[16];
            decode32_f2(q[u], d);
            const float2 s2 = make_float2(s_old[u], s_old[u]);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint32_t gw[4] = {g[u][h].x, g[u][h].y, g[u][h].z, g[u][h].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 gr = make_float2(bf16lo_to_f32(gw[j]), bf16hi_to_f32(gw[j]));
                    d[4 * h + j] = add2_rounded(mul2_rounded(d[4 * h + j], s2), gr);
                }
            }
            const float mx = group_max<LPB>(lane_max_abs(d));
            float qs, m_new;
            agoq_scales(mx, qs, m_new);
            if (valid[u]) {
                uint4 oq[2];
                encode32_f2(d, qs, oq);
                stg128_stream(codes + off[u], oq[0]);
                stg128_stream(codes + off[u] + 16, oq[1]);
                if (part == 0)
                    scale[blk[u]] = m_new;
            }
        }
    }
}

template <typename K> cudaError_t grid_for(K kernel, int64_t lanes_total, int *grid)
{
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBlockThreads, 0);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        per_sm = 1;
    const int64_t need = (lanes_total + kBlockThreads - 1) / kBlockThreads;
    const int64_t cap = static_cast<int64_t>(di.num_sms) * per_sm;
    *grid = static_cast<int>(need < cap ? need : cap);
    return cudaSuccess;
}

// wide: every shard's codes are 32-byte aligned, so a lane of the 32-element
// layout (up to four shards) loads each shard's codes with one 32-byte load.
// With two 16-byte loads each warp request touches 32 sectors half and L2
// serves every sector twice; the wide loads took the headline step from
// 118.9 to 117.9 us (reduce 32.8 -> 31.5 us sampled), measured in one call.
template <int NB, int P>
cudaError_t run_taco_reduce(const ShardPtrs &in, int64_t nblocks, float e_target, float eps,
                            uint8_t *oc, float *oa, float *os, bool wide, cudaStream_t st)
{
    int grid = 0;
    cudaError_t e;
    if constexpr (P <= 4) {
        auto kernel = wide ? taco_reduce_kernel<NB, P, true> : taco_reduce_kernel<NB, P, false>;
        if ((e = grid_for(kernel, nblocks * lanes_per_block<NB, P>(), &grid)) != cudaSuccess)
            return e;
        return launch_pdl(kernel, grid, kBlockThreads, 0, st, in, nblocks, e_target, eps, oc, oa, os);
    } else {
        if ((e = grid_for(taco_reduce_many_kernel<NB, P>, nblocks * lanes_per_block<NB, P>(), &grid)) !=
            cudaSuccess)
            return e;
        return launch_pdl(taco_reduce_many_kernel<NB, P>, grid, kBlockThreads, 0, st, in, nblocks, e_target, eps,
                          oc, oa, os);
    }
}

template <int NB, int P>
cudaError_t run_agoq_reduce(const ShardPtrs &in, int64_t nblocks, uint8_t *oc, float *os, cudaStream_t st)
{
    int grid = 0;
    cudaError_t e = grid_for(agoq_reduce_kernel<NB, P>, nblocks * lanes_per_block<NB, P>(), &grid);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(agoq_reduce_kernel<NB, P>, grid, kBlockThreads, 0, st, in, nblocks, oc, os);
}

template <int NB, int... Ps> struct PDispatch;
template <int NB> struct PDispatch<NB> {
    static cudaError_t taco(int, const ShardPtrs &, int64_t, float, float, uint8_t *, float *, float *, bool,
                            cudaStream_t)
    {
        return cudaErrorInvalidValue;
    }
    static cudaError_t agoq(int, const ShardPtrs &, int64_t, uint8_t *, float *, cudaStream_t)
    {
        return cudaErrorInvalidValue;
    }
};
template <int NB, int P0, int... Ps> struct PDispatch<NB, P0, Ps...> {
    static cudaError_t taco(int P, const ShardPtrs &in, int64_t nb, float e, float eps, uint8_t *oc,
                            float *oa, float *os, bool wide, cudaStream_t st)
    {
        if (P == P0)
            return run_taco_reduce<NB, P0>(in, nb, e, eps, oc, oa, os, wide, st);
        return PDispatch<NB, Ps...>::taco(P, in, nb, e, eps, oc, oa, os, wide, st);
    }
    static cudaError_t agoq(int P, const ShardPtrs &in, int64_t nb, uint8_t *oc, float *os, cudaStream_t st)
    {
        if (P == P0)
            return run_agoq_reduce<NB, P0>(in, nb, oc, os, st);
        return PDispatch<NB, Ps...>::agoq(P, in, nb, oc, os, st);
    }
};

template <int NB>
using AllP = PDispatch<NB, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16>;

}  // namespace

cudaError_t launch_taco_reduce(int P, const ShardPtrs &in, int64_t nblocks, int block, float e_target,
                               float eps, uint8_t *out_codes, float *out_alpha, float *out_scale,
                               cudaStream_t stream)
{
    bool wide = true;
    for (int p = 0; p < P; ++p)
        wide = wide && (reinterpret_cast<uintptr_t>(in.codes[p]) % 32 == 0);
    if (block == 128)
        return AllP<128>::taco(P, in, nblocks, e_target, eps, out_codes, out_alpha, out_scale, wide, stream);
    return AllP<256>::taco(P, in, nblocks, e_target, eps, out_codes, out_alpha, out_scale, wide, stream);
}

// TACO 2.B.3: the rank that reduces both sends the compressed sum (the
// AllGather payload) and uses its reconstruction.  The two kernels run back
// to back on the stream, so the outputs are those of the two separate calls.
// One-pass kernels were built for both block sizes and measured slower in
// the back-to-back step: at n=128 (16-row tiles, two CTAs per SM) the step
// took 127.8 us against 122.5 us, at n=256 (32-row tiles, one CTA per SM)
// the call took 135.5 us against 116.4 us.  A one-pass kernel saves the
// re-read of the compressed sum, but its warps alternate between the
// reduce's load-bound phase and the decompress's store-bound phase, and the
// decompress phase holds registers and staging memory that cap it at 16
// warps per SM.
cudaError_t launch_reduce_decompress(int P, const ShardPtrs &in, int64_t nrows, int block, float e_target,
                                     float eps, uint8_t *out_codes, float *out_alpha, float *out_scale,
                                     void *out, bool out_bf16, cudaStream_t stream)
{
    const cudaError_t e = launch_taco_reduce(P, in, nrows * 128 / block, block, e_target, eps, out_codes,
                                             out_alpha, out_scale, stream);
    if (e != cudaSuccess)
        return e;
    return launch_decompress(out_codes, out_alpha, out_scale, nrows, block, out, out_bf16, false, stream);
}

cudaError_t launch_agoq_reduce(int P, const ShardPtrs &in, int64_t n, int block, uint8_t *out_codes,
                               float *out_scale, cudaStream_t stream)
{
    const int64_t nblocks = n / block;
    if (block == 128)
        return AllP<128>::agoq(P, in, nblocks, out_codes, out_scale, stream);
    return AllP<256>::agoq(P, in, nblocks, out_codes, out_scale, stream);
}

cudaError_t launch_agoq_accumulate(uint8_t *codes, float *scale, const void *grad_bf16, int64_t n,
                                   int block, cudaStream_t stream)
{
    const int64_t nblocks = n / block;
    const uint16_t *g = static_cast<const uint16_t *>(grad_bf16);
    int grid = 0;
    cudaError_t e;
    if (block == 128) {
        if ((e = grid_for(agoq_accumulate_kernel<128>, (nblocks * (128 / kLaneElems) + kAccSlots - 1) / kAccSlots, &grid)) != cudaSuccess)
            return e;
        return launch_pdl(agoq_accumulate_kernel<128>, grid, kBlockThreads, 0, stream, codes, scale, g,
                          nblocks);
    }
    if ((e = grid_for(agoq_accumulate_kernel<256>, (nblocks * (256 / kLaneElems) + kAccSlots - 1) / kAccSlots, &grid)) != cudaSuccess)
        return e;
    return launch_pdl(agoq_accumulate_kernel<256>, grid, kBlockThreads, 0, stream, codes, scale, g, nblocks);
}

}  // namespace taco
