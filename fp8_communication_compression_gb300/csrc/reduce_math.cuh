// Lane-level arithmetic of the shard reductions, shared by the shard-reduce
// kernels and phase 1 of the fused reduce + decompress kernel so that both
// produce bit-identical results.  A lane owns 32 consecutive elements of a
// block (two 16-byte code words per shard) and keeps them as 16 float2
// registers; products and sums use packed fp32x2 instructions, each product
// rounded before it is added (no fused multiply-add).
#pragma once

#include <cfloat>
#include <cstdint>

#include "device_utils.cuh"

namespace taco {

constexpr int kLaneElems = 32;

// 16 E4M3 codes -> 8 float2 (element order), exact.
__device__ __forceinline__ void decode16_f2(const uint4 q, float2 *d)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        e4m3x2_to_f32x2(w[t], d[2 * t].x, d[2 * t].y);
        e4m3x2_to_f32x2(w[t] >> 16, d[2 * t + 1].x, d[2 * t + 1].y);
    }
}

__device__ __forceinline__ void decode32_f2(const uint4 (&q)[2], float2 (&d)[16])
{
    decode16_f2(q[0], d);
    decode16_f2(q[1], d + 8);
}

// 32 values times k -> 32 E4M3 codes (two 16-byte words).
__device__ __forceinline__ void encode32_f2(const float2 (&v)[16], float k, uint4 (&q)[2])
{
    const float2 k2 = make_float2(k, k);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float2 p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            p[i] = __fmul2_rn(v[8 * h + i], k2);
        q[h].x = f32x4_to_e4m3x4(p[0].x, p[0].y, p[1].x, p[1].y);
        q[h].y = f32x4_to_e4m3x4(p[2].x, p[2].y, p[3].x, p[3].y);
        q[h].z = f32x4_to_e4m3x4(p[4].x, p[4].y, p[5].x, p[5].y);
        q[h].w = f32x4_to_e4m3x4(p[6].x, p[6].y, p[7].x, p[7].y);
    }
}

__device__ __forceinline__ void load32_codes(const uint8_t *p, bool valid, uint4 (&q)[2])
{
    q[0] = valid ? ldg128_stream(p) : make_uint4(0, 0, 0, 0);
    q[1] = valid ? ldg128_stream(p + 16) : make_uint4(0, 0, 0, 0);
}

// S = sum_p decode(q_p) * w_p over a compile-time number of shards, in shard
// order; every product is rounded before it is added, so shards that cancel
// exactly sum to exactly zero.
template <int P>
__device__ __forceinline__ void weighted_sum(const uint4 (&q)[P][2], const float (&w)[P], float2 (&S)[16])
{
    decode32_f2(q[0], S);
    const float2 w0 = make_float2(w[0], w[0]);
#pragma unroll
    for (int i = 0; i < 16; ++i)
        S[i] = mul2_rounded(S[i], w0);
#pragma unroll
    for (int p = 1; p < P; ++p) {
        float2 d[16];
        decode32_f2(q[p], d);
        const float2 wp = make_float2(w[p], w[p]);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            S[i] = add2_rounded(S[i], mul2_rounded(d[i], wp));
    }
}

// Adds shard p (p > 0) or starts the sum (p == 0): the run-time-P form of
// weighted_sum, with the same rounding.
__device__ __forceinline__ void weighted_sum_step(const uint4 (&q)[2], float w, bool first, float2 (&S)[16])
{
    float2 d[16];
    decode32_f2(q, d);
    const float2 w2 = make_float2(w, w);
    if (first) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            S[i] = mul2_rounded(d[i], w2);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            S[i] = add2_rounded(S[i], mul2_rounded(d[i], w2));
    }
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

// Largest |value| of the lane's 32 values.
__device__ __forceinline__ float lane_max_abs(const float2 (&S)[16])
{
    float m[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 16; ++i)
        m[i & 1] = fmaxf(m[i & 1], fmaxf(fabsf(S[i].x), fabsf(S[i].y)));
    return fmaxf(m[0], m[1]);
}

// Sum of squares of the lane's 32 values (packed accumulators).
__device__ __forceinline__ float lane_sum_squares(const float2 (&S)[16])
{
    float2 a = __fmul2_rn(S[0], S[0]), b = __fmul2_rn(S[1], S[1]);
#pragma unroll
    for (int i = 2; i < 16; i += 2) {
        a = __ffma2_rn(S[i], S[i], a);
        b = __ffma2_rn(S[i + 1], S[i + 1], b);
    }
    const float2 c = __fadd2_rn(a, b);
    return c.x + c.y;
}

// TACO re-compression of the Hadamard-domain sum T of a block (the lane
// holds 32 of its values; LPB lanes share the block):
//   alpha' = sqrt(E / (|T|^2 / n + eps)),  s' = 448 / (alpha' max|T|),
//   codes  = E4M3(alpha' s' T).
template <int NB, int LPB>
__device__ __forceinline__ void recompress(float2 (&T)[16], float e_target, float eps, uint4 (&codes)[2],
                                           float &alpha, float &scale)
{
    const float ss = group_sum<LPB>(lane_sum_squares(T));
    const float mx = group_max<LPB>(lane_max_abs(T));
    alpha = sqrtf(e_target / (ss * (1.0f / NB) + eps));
    const float M = alpha * mx;
    scale = (M > 0.0f) ? fminf(448.0f / M, FLT_MAX) : 1.0f;
    float k = alpha * scale;
    if (!(k <= FLT_MAX)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            T[i] = __fmul2_rn(T[i], a2);
        k = scale;
    }
    encode32_f2(T, k, codes);
}

// 1 / (s alpha) of shard p's block, the weight of its decoded codes in the
// Hadamard-domain sum (correctly rounded reciprocal; two steps when s alpha
// overflows).
__device__ __forceinline__ float shard_weight(float sc, float al)
{
    const float sa = sc * al;
    return (sa <= FLT_MAX) ? __frcp_rn(sa) : __frcp_rn(sc) / al;
}

}  // namespace taco
