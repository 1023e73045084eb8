// Lane-level arithmetic of the shard reductions, shared by the shard-reduce
// kernels, the AGoQ accumulate kernel and the AGoQ epilogue of the GEMM.  A lane owns 16 or 32 consecutive
// elements of a block (one or two 16-byte code words per shard), kept as
// NF = 8 or 16 float2 registers; the block statistics are bit-identical in
// either layout.  The
// weighted sums round every product before adding it (scalar __fmul_rn /
// __fadd_rn, never contracted into a fused multiply-add); the statistics and
// the re-encoding use packed fp32x2 instructions.
#pragma once

#include <cfloat>
#include <cstdint>

#include "device_utils.cuh"

namespace taco {

constexpr int kLaneElems = 32;  // elements per lane in the default layout

// A lane holds NF float2 registers: 16 (32 elements) or 8 (16 elements).
// Everything below is written so that a block's statistics come out
// bit-identical in either layout.

// 4 E4M3 codes (bytes 0..3 of w) -> 2 float2, exact: the word's two halves
// go to the FP8-pair conversion as register halves, with no shift.
__device__ __forceinline__ void decode4_f2(uint32_t w, float2 &a, float2 &b)
{
    uint32_t h0, h1;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
    asm("{\n\t.reg .f16 a, b, c, d;\n\tmov.b32 {a, b}, %4;\n\tmov.b32 {c, d}, %5;\n\t"
        "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\tcvt.f32.f16 %2, c;\n\tcvt.f32.f16 %3, d;\n\t}"
        : "=f"(a.x), "=f"(a.y), "=f"(b.x), "=f"(b.y)
        : "r"(h0), "r"(h1));
}

// 16 E4M3 codes -> 8 float2 (element order), exact.
__device__ __forceinline__ void decode16_f2(const uint4 q, float2 *d)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t)
        decode4_f2(w[t], d[2 * t], d[2 * t + 1]);
}

template <int NF> __device__ __forceinline__ void decode_codes(const uint4 (&q)[NF / 8], float2 (&d)[NF])
{
#pragma unroll
    for (int h = 0; h < NF / 8; ++h)
        decode16_f2(q[h], d + 8 * h);
}

__device__ __forceinline__ void decode32_f2(const uint4 (&q)[2], float2 (&d)[16]) { decode_codes<16>(q, d); }

// NF float2 values times k -> E4M3 codes (NF / 8 16-byte words).
template <int NF> __device__ __forceinline__ void encode_codes(const float2 (&v)[NF], float k, uint4 (&q)[NF / 8])
{
    const float2 k2 = make_float2(k, k);
#pragma unroll
    for (int h = 0; h < NF / 8; ++h) {
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

__device__ __forceinline__ void encode32_f2(const float2 (&v)[16], float k, uint4 (&q)[2]) { encode_codes<16>(v, k, q); }

// 32 codes with one 32-byte load (p 32-byte aligned) and an L2 cache
// policy: a warp's request then covers 32 whole sectors, where two 16-byte
// loads 32 bytes apart each touch 32 sectors half.
__device__ __forceinline__ void ldg256_stream_hint(const void *p, uint64_t pol, uint4 &lo, uint4 &hi)
{
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p), "l"(pol));
}

// EF: load with the L2 cache policy `pol` (evict-first for codes that
// nothing reads again); without EF, `pol` is ignored.  WIDE (32 codes, EF,
// p 32-byte aligned): one 32-byte load instead of two 16-byte ones.
template <int NF, bool EF = false, bool WIDE = false>
__device__ __forceinline__ void load_codes(const uint8_t *p, bool valid, uint4 (&q)[NF / 8], uint64_t pol = 0)
{
    if constexpr (WIDE) {
        static_assert(NF == 16 && EF, "the 32-byte load covers 32 codes, with a cache policy");
        if (valid) {
            ldg256_stream_hint(p, pol, q[0], q[1]);
        } else {
            q[0] = make_uint4(0, 0, 0, 0);
            q[1] = make_uint4(0, 0, 0, 0);
        }
    } else {
#pragma unroll
        for (int h = 0; h < NF / 8; ++h) {
            if (!valid)
                q[h] = make_uint4(0, 0, 0, 0);
            else if constexpr (EF)
                q[h] = ldg128_stream_hint(p + 16 * h, pol);
            else
                q[h] = ldg128_stream(p + 16 * h);
        }
    }
}

// S = sum_p decode(q_p) * w_p over a compile-time number of shards, in shard
// order.  Every product is rounded before it is added (__fmul_rn / __fadd_rn
// are never contracted into a fused multiply-add), so shards that cancel
// exactly sum to exactly zero.
template <int P, int NF>
__device__ __forceinline__ void weighted_sum(const uint4 (&q)[P][NF / 8], const float (&w)[P], float2 (&S)[NF])
{
    decode_codes<NF>(q[0], S);
    const float2 w0 = make_float2(w[0], w[0]);
#pragma unroll
    for (int i = 0; i < NF; ++i)
        S[i] = mul2_rounded(S[i], w0);
#pragma unroll
    for (int p = 1; p < P; ++p) {
        float2 d[NF];
        decode_codes<NF>(q[p], d);
        const float2 wp = make_float2(w[p], w[p]);
#pragma unroll
        for (int i = 0; i < NF; ++i)
            S[i] = add2_rounded(S[i], mul2_rounded(d[i], wp));
    }
}

// Sum over the LPB lanes of a group.  The xor butterfly runs in ascending
// order (1, 2, 4, ...), which adds aligned neighbours first: with partial
// sums p_0, p_1, ... in element order the result is the balanced tree
// ((p_0 + p_1) + (p_2 + p_3)) + ..., whatever the number of partials per
// lane (floating-point addition is commutative).
template <int LPB> __device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = 1; o < LPB; o <<= 1)
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

// Largest |value| of the lane's values.
template <int NF> __device__ __forceinline__ float lane_max_abs(const float2 (&S)[NF])
{
    float m[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < NF; ++i)
        m[i & 1] = fmaxf(m[i & 1], fmaxf(fabsf(S[i].x), fabsf(S[i].y)));
    return fmaxf(m[0], m[1]);
}

// Sum of squares of 16 consecutive elements (8 float2), in one fixed order.
__device__ __forceinline__ float sum_squares16(const float2 *S)
{
    float2 a = __fmul2_rn(S[0], S[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i)
        a = __ffma2_rn(S[i], S[i], a);
    return a.x + a.y;
}

// The lane's share of the block's sum of squares: its 16-element partials
// added in pairs (see group_sum for how the lanes' shares combine).
template <int NF> __device__ __forceinline__ float lane_sum_squares(const float2 (&S)[NF])
{
    if constexpr (NF == 8)
        return sum_squares16(S);
    else
        return sum_squares16(S) + sum_squares16(S + 8);
}

// TACO re-compression of the Hadamard-domain sum T of a block (the lane
// holds 2 NF of its values; LPB lanes share the block):
//   alpha' = sqrt(E / (|T|^2 / n + eps)),  s' = 448 / (alpha' max|T|),
//   codes  = E4M3(alpha' s' T).
template <int NB, int LPB, int NF>
__device__ __forceinline__ void recompress(float2 (&T)[NF], float e_target, float eps, uint4 (&codes)[NF / 8],
                                           float &alpha, float &scale)
{
    const float ss = group_sum<LPB>(lane_sum_squares<NF>(T));
    const float mx = group_max<LPB>(lane_max_abs<NF>(T));
    alpha = sqrtf(e_target / (ss * (1.0f / NB) + eps));
    const float M = alpha * mx;
    scale = (M > 0.0f) ? fminf(448.0f / M, FLT_MAX) : 1.0f;
    float k = alpha * scale;
    if (!(k <= FLT_MAX)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < NF; ++i)
            T[i] = __fmul2_rn(T[i], a2);
        k = scale;
    }
    encode_codes<NF>(T, k, codes);
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

// 1 / (s alpha) of shard p's block, the weight of its decoded codes in the
// Hadamard-domain sum (correctly rounded reciprocal; two steps when s alpha
// overflows).
__device__ __forceinline__ float shard_weight(float sc, float al)
{
    const float sa = sc * al;
    return (sa <= FLT_MAX) ? __frcp_rn(sa) : __frcp_rn(sc) / al;
}

}  // namespace taco
