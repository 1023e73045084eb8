// Shard reduce (TACO two-shot local step) and AGoQ FP8 gradient kernels for
// sm_103a.  None of these needs a Hadamard rotation on its path, so they
// use plain coalesced 16-byte loads: a lane owns 32 consecutive elements of
// a block, NB / 32 adjacent lanes own one block, per-block statistics (sum
// of squares, absolute maximum) are combined with __shfl_xor_sync, and the
// per-shard scalars of a block are fetched once per lane group and
// broadcast with __shfl_sync.
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

namespace taco {

namespace {

constexpr int kEPL = 32;  // elements per lane
constexpr int kBlockThreads = 256;

// 32 codes (two 16-byte words) -> 32 fp32 values (exact)
__device__ __forceinline__ void decode32(const uint4 (&q)[2], float (&d)[32])
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w[4] = {q[h].x, q[h].y, q[h].z, q[h].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            e4m3x2_to_f32x2(w[j], d[16 * h + 4 * j + 0], d[16 * h + 4 * j + 1]);
            e4m3x2_to_f32x2(w[j] >> 16, d[16 * h + 4 * j + 2], d[16 * h + 4 * j + 3]);
        }
    }
}

__device__ __forceinline__ void encode32(const float (&v)[32], float k, uint4 (&q)[2])
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float *x = v + 16 * h;
        q[h].x = f32x4_to_e4m3x4(x[0] * k, x[1] * k, x[2] * k, x[3] * k);
        q[h].y = f32x4_to_e4m3x4(x[4] * k, x[5] * k, x[6] * k, x[7] * k);
        q[h].z = f32x4_to_e4m3x4(x[8] * k, x[9] * k, x[10] * k, x[11] * k);
        q[h].w = f32x4_to_e4m3x4(x[12] * k, x[13] * k, x[14] * k, x[15] * k);
    }
}

__device__ __forceinline__ void load32_codes(const uint8_t *p, bool valid, uint4 (&q)[2])
{
    q[0] = valid ? ldg128_stream(p) : make_uint4(0, 0, 0, 0);
    q[1] = valid ? ldg128_stream(p + 16) : make_uint4(0, 0, 0, 0);
}

template <int LPB> __device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = LPB / 2; o >= 1; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

template <int LPB> __device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = LPB / 2; o >= 1; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// AGoQ per-block requantisation scalars from the block's absolute maximum:
// codes use q = 448 / amax; the stored scale is the dequantisation
// multiplier m = amax / 448 (both 1 for an all-zero block).
__device__ __forceinline__ void agoq_scales(float amax, float &q, float &m)
{
    if (amax > 0.0f) {
        q = fminf(448.0f / amax, FLT_MAX);
        m = amax / 448.0f;
    } else {
        q = 1.0f;
        m = 1.0f;
    }
}

// Warp-uniform grid-stride loop over lane slots.  Lanes past the end still
// take part in the shuffles but load and store nothing.
#define TACO_LANE_LOOP(total)                                                                    \
    pdl_wait();                                                                                  \
    pdl_launch_dependents();                                                                     \
    const int64_t _stride = static_cast<int64_t>(gridDim.x) * blockDim.x;                        \
    for (int64_t _base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);    \
         _base < (total); _base += _stride)

// ------------------------------------------------------ TACO reduce --

template <int NB, int P>
__global__ void __launch_bounds__(kBlockThreads)
    taco_reduce_kernel(const ShardPtrs in, int64_t nblocks, float e_target, float eps,
                       uint8_t *__restrict__ out_codes, float *__restrict__ out_alpha,
                       float *__restrict__ out_scale)
{
    constexpr int LPB = NB / kEPL;
    const int64_t total = nblocks * LPB;
    const int lane = threadIdx.x & 31;
    TACO_LANE_LOOP(total)
    {
        const int64_t t = _base + lane;
        const bool valid = t < total;
        const int64_t blk = valid ? t / LPB : 0;
        const int part = static_cast<int>(t % LPB);
        const int64_t off = blk * NB + part * kEPL;
        uint4 q[P][2];
#pragma unroll
        for (int p = 0; p < P; ++p)
            load32_codes(in.codes[p] + off, valid, q[p]);
        // 1 / (s_p alpha_p): lane `part` of the group computes it for shards
        // part, part + LPB, ...; the group then shares the values.
        constexpr int ROUNDS = (P + LPB - 1) / LPB;
        float wr[ROUNDS];
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
            const int p = r * LPB + part;
            wr[r] = 1.0f;
            if (valid && p < P) {
                const float sc = __ldg(in.scale[p] + blk), al = __ldg(in.alpha[p] + blk);
                const float sa = sc * al;
                wr[r] = (sa <= FLT_MAX) ? __frcp_rn(sa) : __frcp_rn(sc) / al;
            }
        }
        const int gbase = lane & ~(LPB - 1);
        float w[P];
#pragma unroll
        for (int p = 0; p < P; ++p)
            w[p] = __shfl_sync(0xFFFFFFFFu, wr[p / LPB], gbase + (p % LPB));
        // Each product is rounded before it is added (no FMA contraction), so
        // shards that cancel exactly sum to exactly zero.
        float T[kEPL];
        decode32(q[0], T);
#pragma unroll
        for (int i = 0; i < kEPL; ++i)
            T[i] = __fmul_rn(T[i], w[0]);
#pragma unroll
        for (int p = 1; p < P; ++p) {
            float d[kEPL];
            decode32(q[p], d);
#pragma unroll
            for (int i = 0; i < kEPL; ++i)
                T[i] = __fadd_rn(T[i], __fmul_rn(d[i], w[p]));
        }
        float a4[4] = {0.f, 0.f, 0.f, 0.f}, mx = 0.0f;
#pragma unroll
        for (int i = 0; i < kEPL; ++i) {
            a4[i & 3] = fmaf(T[i], T[i], a4[i & 3]);
            mx = fmaxf(mx, fabsf(T[i]));
        }
        const float ss = group_sum<LPB>((a4[0] + a4[1]) + (a4[2] + a4[3]));
        mx = group_max<LPB>(mx);
        const float alpha = sqrtf(e_target / (ss * (1.0f / NB) + eps));
        const float M = alpha * mx;
        const float scale = (M > 0.0f) ? fminf(448.0f / M, FLT_MAX) : 1.0f;
        float k = alpha * scale;
        if (!(k <= FLT_MAX)) {
#pragma unroll
            for (int i = 0; i < kEPL; ++i)
                T[i] *= alpha;
            k = scale;
        }
        if (valid) {
            uint4 oq[2];
            encode32(T, k, oq);
            stg128_stream(out_codes + off, oq[0]);
            stg128_stream(out_codes + off + 16, oq[1]);
            if (part == 0) {
                out_alpha[blk] = alpha;
                out_scale[blk] = scale;
            }
        }
    }
}

// ------------------------------------------------- AGoQ accumulate --

template <int NB>
__global__ void __launch_bounds__(kBlockThreads)
    agoq_accumulate_kernel(uint8_t *__restrict__ codes, float *__restrict__ scale,
                           const uint16_t *__restrict__ grad, int64_t nblocks)
{
    constexpr int LPB = NB / kEPL;
    const int64_t total = nblocks * LPB;
    const int lane = threadIdx.x & 31;
    TACO_LANE_LOOP(total)
    {
        const int64_t t = _base + lane;
        const bool valid = t < total;
        const int64_t blk = valid ? t / LPB : 0;
        const int part = static_cast<int>(t % LPB);
        const int64_t off = blk * NB + part * kEPL;
        uint4 q[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        uint4 g[4] = {q[0], q[0], q[0], q[0]};
        float s_old = 1.0f;
        if (valid) {
            // codes and scale are rewritten below: coherent loads, not .nc
#pragma unroll
            for (int h = 0; h < 2; ++h)
                asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(q[h].x), "=r"(q[h].y), "=r"(q[h].z), "=r"(q[h].w)
                             : "l"(codes + off + 16 * h));
#pragma unroll
            for (int h = 0; h < 4; ++h)
                g[h] = ldg128_stream(grad + off + 8 * h);
            asm volatile("ld.global.f32 %0, [%1];" : "=f"(s_old) : "l"(scale + blk));
        }
        // g = dequantise(main) + grad in FP32: one rounded multiply, then one
        // rounded add (no fused multiply-add), as the stated arithmetic is.
        float d[kEPL];
        decode32(q, d);
        float mx = 0.0f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint32_t gw[4] = {g[h].x, g[h].y, g[h].z, g[h].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = 8 * h + 2 * j;
                d[e] = __fadd_rn(__fmul_rn(d[e], s_old), bf16lo_to_f32(gw[j]));
                d[e + 1] = __fadd_rn(__fmul_rn(d[e + 1], s_old), bf16hi_to_f32(gw[j]));
                mx = fmaxf(mx, fmaxf(fabsf(d[e]), fabsf(d[e + 1])));
            }
        }
        mx = group_max<LPB>(mx);
        float qs, m_new;
        agoq_scales(mx, qs, m_new);
        if (valid) {
            uint4 oq[2];
            encode32(d, qs, oq);
            stg128_stream(codes + off, oq[0]);
            stg128_stream(codes + off + 16, oq[1]);
            if (part == 0)
                scale[blk] = m_new;
        }
    }
}

// ----------------------------------------------------- AGoQ reduce --

template <int NB, int P>
__global__ void __launch_bounds__(kBlockThreads)
    agoq_reduce_kernel(const ShardPtrs in, int64_t nblocks, uint8_t *__restrict__ out_codes,
                       float *__restrict__ out_scale)
{
    constexpr int LPB = NB / kEPL;
    const int64_t total = nblocks * LPB;
    const int lane = threadIdx.x & 31;
    TACO_LANE_LOOP(total)
    {
        const int64_t t = _base + lane;
        const bool valid = t < total;
        const int64_t blk = valid ? t / LPB : 0;
        const int part = static_cast<int>(t % LPB);
        const int64_t off = blk * NB + part * kEPL;
        uint4 q[P][2];
#pragma unroll
        for (int p = 0; p < P; ++p)
            load32_codes(in.codes[p] + off, valid, q[p]);
        constexpr int ROUNDS = (P + LPB - 1) / LPB;
        float mr[ROUNDS];
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
            const int p = r * LPB + part;
            mr[r] = (valid && p < P) ? __ldg(in.scale[p] + blk) : 1.0f;
        }
        const int gbase = lane & ~(LPB - 1);
        float m[P];
#pragma unroll
        for (int p = 0; p < P; ++p)
            m[p] = __shfl_sync(0xFFFFFFFFu, mr[p / LPB], gbase + (p % LPB));
        // FP32 dequantise (one rounded multiply) and FP32 sum in shard order,
        // no fused multiply-add: exactly cancelling shards give exactly 0
        float S[kEPL];
        decode32(q[0], S);
#pragma unroll
        for (int i = 0; i < kEPL; ++i)
            S[i] = __fmul_rn(S[i], m[0]);
#pragma unroll
        for (int p = 1; p < P; ++p) {
            float d[kEPL];
            decode32(q[p], d);
#pragma unroll
            for (int i = 0; i < kEPL; ++i)
                S[i] = __fadd_rn(S[i], __fmul_rn(d[i], m[p]));
        }
        float mx = 0.0f;
#pragma unroll
        for (int i = 0; i < kEPL; ++i)
            mx = fmaxf(mx, fabsf(S[i]));
        mx = group_max<LPB>(mx);
        float qs, m_new;
        agoq_scales(mx, qs, m_new);
        if (valid) {
            uint4 oq[2];
            encode32(S, qs, oq);
            stg128_stream(out_codes + off, oq[0]);
            stg128_stream(out_codes + off + 16, oq[1]);
            if (part == 0)
                out_scale[blk] = m_new;
        }
    }
}

#undef TACO_LANE_LOOP

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

template <int NB, int P>
cudaError_t run_taco_reduce(const ShardPtrs &in, int64_t nblocks, float e_target, float eps,
                            uint8_t *oc, float *oa, float *os, cudaStream_t st)
{
    int grid = 0;
    cudaError_t e = grid_for(taco_reduce_kernel<NB, P>, nblocks * (NB / kEPL), &grid);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(taco_reduce_kernel<NB, P>, grid, kBlockThreads, 0, st, in, nblocks, e_target, eps, oc,
                      oa, os);
}

template <int NB, int P>
cudaError_t run_agoq_reduce(const ShardPtrs &in, int64_t nblocks, uint8_t *oc, float *os, cudaStream_t st)
{
    int grid = 0;
    cudaError_t e = grid_for(agoq_reduce_kernel<NB, P>, nblocks * (NB / kEPL), &grid);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(agoq_reduce_kernel<NB, P>, grid, kBlockThreads, 0, st, in, nblocks, oc, os);
}

template <int NB, int... Ps> struct PDispatch;
template <int NB> struct PDispatch<NB> {
    static cudaError_t taco(int, const ShardPtrs &, int64_t, float, float, uint8_t *, float *, float *,
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
                            float *oa, float *os, cudaStream_t st)
    {
        if (P == P0)
            return run_taco_reduce<NB, P0>(in, nb, e, eps, oc, oa, os, st);
        return PDispatch<NB, Ps...>::taco(P, in, nb, e, eps, oc, oa, os, st);
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
    if (block == 128)
        return AllP<128>::taco(P, in, nblocks, e_target, eps, out_codes, out_alpha, out_scale, stream);
    return AllP<256>::taco(P, in, nblocks, e_target, eps, out_codes, out_alpha, out_scale, stream);
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
        if ((e = grid_for(agoq_accumulate_kernel<128>, nblocks * (128 / kEPL), &grid)) != cudaSuccess)
            return e;
        e = launch_pdl(agoq_accumulate_kernel<128>, grid, kBlockThreads, 0, stream, codes, scale, g, nblocks);
    } else {
        if ((e = grid_for(agoq_accumulate_kernel<256>, nblocks * (256 / kEPL), &grid)) != cudaSuccess)
            return e;
        e = launch_pdl(agoq_accumulate_kernel<256>, grid, kBlockThreads, 0, stream, codes, scale, g, nblocks);
    }
    return e;
}

}  // namespace taco
