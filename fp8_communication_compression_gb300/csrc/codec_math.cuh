// Row arithmetic shared by the codec kernels: a thread holds one 128-element
// row of a block in 64 float2 registers and runs the Walsh-Hadamard
// butterflies, the block statistics and the E4M3 conversions on it.
#pragma once

#include <cfloat>
#include <cstdint>

#include "device_utils.cuh"

namespace taco {

template <int NB> struct BlockConst;
template <> struct BlockConst<128> {
    static constexpr float c = 0.0883883461356163f;  // fp32(1/sqrt(128))
    static constexpr float inv_n = 1.0f / 128.0f;
};
template <> struct BlockConst<256> {
    static constexpr float c = 0.0625f;              // 1/sqrt(256), exact
    static constexpr float inv_n = 1.0f / 256.0f;
};

// A thread's 128-element row lives in 64 float2 registers: v[k] holds
// elements 2k and 2k + 1.  The butterfly stage on index bit 0 is done with
// scalar adds while the row is unpacked; the stages on bits 1..6 pair whole
// float2 registers and run as packed fp32x2 instructions (sm_100 family),
// which halves their instruction count.  a - b is computed as
// fma(b, -1, a): the product is exact, so the result (signed zeros
// included) is that of the subtraction.

__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}

// Stages h = 2, 4, ..., 64 of the unnormalised Sylvester-order Walsh-
// Hadamard transform: pairs (i, i + h) become (a + b, a - b).  Together
// with the bit-0 stage done at unpack time this is the full 128-point
// transform, in the order h = 1, 2, ..., 64.
__device__ __forceinline__ void fwht128_upper(float2 (&v)[64])
{
#pragma unroll
    for (int hh = 1; hh < 64; hh <<= 1) {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
            if ((k & hh) == 0) {
                const float2 a = v[k], b = v[k + hh];
                v[k] = __fadd2_rn(a, b);
                v[k + hh] = sub2(a, b);
            }
        }
    }
}

// Stages h = 2, 4, ..., 32: all but the last stage of the 128-point
// transform (which pairs v[k] with v[k + 32]).
__device__ __forceinline__ void fwht128_upper_but_last(float2 (&v)[64])
{
#pragma unroll
    for (int hh = 1; hh < 32; hh <<= 1) {
#pragma unroll
        for (int k = 0; k < 64; ++k) {
            if ((k & hh) == 0) {
                const float2 a = v[k], b = v[k + hh];
                v[k] = __fadd2_rn(a, b);
                v[k + hh] = sub2(a, b);
            }
        }
    }
}

__device__ __forceinline__ float2 abs2(float2 a) { return make_float2(fabsf(a.x), fabsf(a.y)); }

// Largest |y| of the full transform, read off the operands of its last
// stage: max(|a + b|, |a - b|) = |a| + |b|, and fp32 rounding keeps the
// identity (|round(a + b)| and |round(a - b)| are round(|a| + |b|) and a
// smaller value).
__device__ __forceinline__ float max_abs_last_stage(const float2 (&v)[64])
{
    float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const float2 t = __fadd2_rn(abs2(v[k]), abs2(v[k + 32]));
        m[k & 3] = fmaxf(m[k & 3], fmaxf(t.x, t.y));
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// The last stage fused with the multiply by k: v[k] <- (a + b) k and
// v[k + 32] <- (a - b) k, as fma(b, +-k, a k).
__device__ __forceinline__ void last_stage_scaled(float2 (&v)[64], float2 k2)
{
    const float2 nk2 = make_float2(-k2.x, -k2.y);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const float2 ak = __fmul2_rn(v[k], k2);
        const float2 b = v[k + 32];
        v[k] = __ffma2_rn(b, k2, ak);
        v[k + 32] = __ffma2_rn(b, nk2, ak);
    }
}

// Last stage of a 256-point transform across a lane pair: the even lane
// holds elements 0..127 (a), the odd lane 128..255 (b); even gets a + b,
// odd gets a - b.
__device__ __forceinline__ void fwht_pair_stage(float2 (&v)[64], int lane)
{
    const float sg = (lane & 1) ? -1.0f : 1.0f;
    const float2 sgn = make_float2(sg, sg);
#pragma unroll
    for (int k = 0; k < 64; ++k) {
        float2 o;
        o.x = __shfl_xor_sync(0xFFFFFFFFu, v[k].x, 1);
        o.y = __shfl_xor_sync(0xFFFFFFFFu, v[k].y, 1);
        v[k] = __ffma2_rn(sgn, v[k], o);
    }
}

__device__ __forceinline__ float max_abs128(const float2 (&v)[64])
{
    float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 64; ++k)
        m[k & 3] = fmaxf(m[k & 3], fmaxf(fabsf(v[k].x), fabsf(v[k].y)));
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// Unpacks 8 bf16 values (one 16-byte chunk) into four float2 registers
// v[k0 .. k0+3] after the bit-0 butterfly stage, and adds their squares to
// the packed energy accumulators.
__device__ __forceinline__ void unpack8_stage1(const uint4 q, float2 (&v)[64], int k0, float2 (&acc)[8],
                                               bool first)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float lo = bf16lo_to_f32(w[t]), hi = bf16hi_to_f32(w[t]);
        const float2 x = make_float2(lo, hi);
        const int a = (k0 + t) & 7;
        acc[a] = first ? __fmul2_rn(x, x) : __ffma2_rn(x, x, acc[a]);
        v[k0 + t] = make_float2(lo + hi, lo - hi);
    }
}

// Four float2 pairs (already scaled) -> 8 E4M3 codes in two words.
__device__ __forceinline__ void encode8_prescaled(const float2 *v, uint32_t &w0, uint32_t &w1)
{
    w0 = f32x4_to_e4m3x4(v[0].x, v[0].y, v[1].x, v[1].y);
    w1 = f32x4_to_e4m3x4(v[2].x, v[2].y, v[3].x, v[3].y);
}

// Four float2 pairs times k -> 8 E4M3 codes in two words.
__device__ __forceinline__ void encode8(const float2 *v, float2 k2, uint32_t &w0, uint32_t &w1)
{
    const float2 a = __fmul2_rn(v[0], k2), b = __fmul2_rn(v[1], k2);
    const float2 c = __fmul2_rn(v[2], k2), d = __fmul2_rn(v[3], k2);
    w0 = f32x4_to_e4m3x4(a.x, a.y, b.x, b.y);
    w1 = f32x4_to_e4m3x4(c.x, c.y, d.x, d.y);
}

// ---- INT8 codes (the fallback format for hardware without native FP8) ----

// Four fp32 values (already scaled into [-127, 127]) -> four int8 codes,
// round to nearest even, packed little-endian.
// Four values already in [-127.5, 127.5) -> four int8 codes, rounded to
// nearest even.  Adding 1.5 * 2^23 rounds a value to an integer in the low
// mantissa bits (the float's unit in the last place is 1 there), and since
// the low byte of 1.5 * 2^23 is zero, that byte is the two's-complement code.
__device__ __forceinline__ uint32_t f32x4_to_s8x4(float a, float b, float c, float d)
{
    const float2 magic = make_float2(12582912.0f, 12582912.0f);
    const float2 p = __fadd2_rn(make_float2(a, b), magic), q = __fadd2_rn(make_float2(c, d), magic);
    const uint32_t lo = __byte_perm(__float_as_uint(p.x), __float_as_uint(p.y), 0x0040);
    const uint32_t hi = __byte_perm(__float_as_uint(q.x), __float_as_uint(q.y), 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

__device__ __forceinline__ void encode8_s8_prescaled(const float2 *v, uint32_t &w0, uint32_t &w1)
{
    w0 = f32x4_to_s8x4(v[0].x, v[0].y, v[1].x, v[1].y);
    w1 = f32x4_to_s8x4(v[2].x, v[2].y, v[3].x, v[3].y);
}

__device__ __forceinline__ void encode8_s8(const float2 *v, float2 k2, uint32_t &w0, uint32_t &w1)
{
    const float2 a = __fmul2_rn(v[0], k2), b = __fmul2_rn(v[1], k2);
    const float2 c = __fmul2_rn(v[2], k2), d = __fmul2_rn(v[3], k2);
    w0 = f32x4_to_s8x4(a.x, a.y, b.x, b.y);
    w1 = f32x4_to_s8x4(c.x, c.y, d.x, d.y);
}

// Four int8 codes -> four fp32 values, exactly: the biased byte b + 128 is
// placed in the low mantissa bits of 2^23, and 2^23 + 128 is subtracted.
__device__ __forceinline__ void s8x4_to_f32x4(uint32_t w, float2 &lo, float2 &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    const float2 bias = make_float2(8388736.0f, 8388736.0f);
    const float2 a = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)),
                                 __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)));
    const float2 b = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)),
                                 __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)));
    lo = __fadd2_rn(a, make_float2(-bias.x, -bias.y));
    hi = __fadd2_rn(b, make_float2(-bias.x, -bias.y));
}

// Decodes one 16-byte chunk of 16 INT8 codes into v[8 j .. 8 j + 7] after
// the bit-0 butterfly stage.
__device__ __forceinline__ void decode16_stage1_s8(const uint4 q, float2 (&v)[64], int j)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        float2 e01, e23;
        s8x4_to_f32x4(w[t], e01, e23);
        v[8 * j + 2 * t] = make_float2(e01.x + e01.y, e01.x - e01.y);
        v[8 * j + 2 * t + 1] = make_float2(e23.x + e23.y, e23.x - e23.y);
    }
}

// Decodes one 16-byte chunk of 16 codes (row elements 16 j .. 16 j + 15)
// into v[8 j .. 8 j + 7] after the bit-0 butterfly stage.
__device__ __forceinline__ void decode16_stage1(const uint4 q, float2 (&v)[64], int j)
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        float e0, e1, e2, e3;
        e4m3x2_to_f32x2(w[t], e0, e1);
        e4m3x2_to_f32x2(w[t] >> 16, e2, e3);
        v[8 * j + 2 * t] = make_float2(e0 + e1, e0 - e1);
        v[8 * j + 2 * t + 1] = make_float2(e2 + e3, e2 - e3);
    }
}

// Decompression multiplier c / (s alpha).  For extreme scales (s alpha
// overflows, or the quotient underflows) the row is divided by s first and
// c / alpha is returned instead.
template <int NB>
__device__ __forceinline__ float2 decompress_multiplier(float2 (&v)[64], float sc, float a)
{
    const float c = BlockConst<NB>::c;
    const float sa = sc * a;
    float k = c / sa;
    if (!(sa <= FLT_MAX) || !(k >= FLT_MIN)) {
        const float inv_s = 1.0f / sc;
        const float2 i2 = make_float2(inv_s, inv_s);
#pragma unroll
        for (int i = 0; i < 64; ++i)
            v[i] = __fmul2_rn(v[i], i2);
        k = c / a;
    }
    return make_float2(k, k);
}

// Writes a row of 128 reconstructed values times k2 into a warp's swizzled
// staging area: fp32 as 4 boxes of 32 floats x 32 rows, or bf16 as 2 boxes
// of 64 values x 32 rows (each box 4 KB, row `lane` at lane * 128 bytes).
// With PRESCALED the values already include the factor and k2 is ignored.
template <bool BF16OUT, bool PRESCALED = false>
__device__ __forceinline__ void stage_output_row(const float2 (&v)[64], float2 k2, uint32_t outw, int lane)
{
    const uint32_t swz = static_cast<uint32_t>(lane & 7) << 4;
    if constexpr (!BF16OUT) {
#pragma unroll
        for (int ch = 0; ch < 32; ++ch) {
            const uint32_t b = ch >> 3, j = ch & 7;
            const uint32_t addr = outw + b * 4096 + lane * 128 + ((j << 4) ^ swz);
            const float2 p0 = PRESCALED ? v[2 * ch] : __fmul2_rn(v[2 * ch], k2);
            const float2 p1 = PRESCALED ? v[2 * ch + 1] : __fmul2_rn(v[2 * ch + 1], k2);
            sts128(addr, __float_as_uint(p0.x), __float_as_uint(p0.y), __float_as_uint(p1.x),
                   __float_as_uint(p1.y));
        }
    } else {
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
            const uint32_t b = ch >> 3, j = ch & 7;
            const uint32_t addr = outw + b * 4096 + lane * 128 + ((j << 4) ^ swz);
            float2 p[4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                p[t] = PRESCALED ? v[4 * ch + t] : __fmul2_rn(v[4 * ch + t], k2);
            sts128(addr, f32x2_to_bf16x2(p[0].x, p[0].y), f32x2_to_bf16x2(p[1].x, p[1].y),
                   f32x2_to_bf16x2(p[2].x, p[2].y), f32x2_to_bf16x2(p[3].x, p[3].y));
        }
    }
}

}  // namespace taco
