// Block-wise activation codec of AGoQ's layer-aware activation quantisation
// (AGoQ, gist.science summary of arXiv 2605.00539, 2.A): activations of the
// quantised layers are stored per block as symmetric b-bit integers (b = 4,
// or 5 / 6 / 8 where the pipeline-stage bit-width compensation grants more
// memory) with one fp32 multiplier per block.
//
// Per block: amax = max|x|, qmax = 2^(b-1) - 1, q = qmax / amax,
// code = clamp(rint(x * q), -qmax, qmax), m = amax / qmax (1 for a zero
// block), x_hat = code * m, all in fp32 with every operation rounded.  Codes
// are two's complement in a little-endian bit stream: element i occupies
// bits i*b .. i*b + b - 1.
//
// The clamp never binds (|x q| <= qmax up to one rounding); the kernels
// round with a magic-number addition instead of conversion instructions.
//
// In the quantizer a lane owns 32 consecutive elements of a block; their 32
// codes are exactly b 32-bit words of the stream, packed with compile-time
// shifts.  Each lane takes several grid-stride slots per loop trip and
// issues all of their loads before it processes the first.  The
// dequantizer's layout is described above its kernel.

#include <cfloat>

#include "device_utils.cuh"
#include "internal.h"
#include "laaq_math.cuh"
#include "reduce_math.cuh"

namespace taco {

namespace {

constexpr int kLThreads = 256;

// The lane's BITS words go to byte offset 4 * BITS * (lane slot): 16-byte
// aligned for 4 and 8 bits, 8-byte for 6, 4-byte for 5.
template <int BITS> __device__ __forceinline__ void store_words(uint8_t *dst, const uint32_t (&w)[BITS])
{
    if constexpr (BITS % 4 == 0) {
#pragma unroll
        for (int j = 0; j < BITS; j += 4)
            stg128_stream(dst + 4 * j, make_uint4(w[j], w[j + 1], w[j + 2], w[j + 3]));
    } else if constexpr (BITS % 2 == 0) {
#pragma unroll
        for (int j = 0; j < BITS; j += 2)
            *reinterpret_cast<uint2 *>(dst + 4 * j) = make_uint2(w[j], w[j + 1]);
    } else {
#pragma unroll
        for (int j = 0; j < BITS; ++j)
            reinterpret_cast<uint32_t *>(dst)[j] = w[j];
    }
}

// Slots a lane loads before it processes any of them: the loads of both
// slots (128 bytes of bf16 per lane) are in flight together.
constexpr int kQuantSlots = 2;

// A lane's 32 bf16 values are 64 contiguous bytes, and lane l's follow lane
// l - 1's.  WIDE (x 32-byte aligned): two 32-byte loads, each filling whole
// 32-byte sectors (lane l reads sector 2l, then 2l + 1), so every sector is
// requested once.  Otherwise four 16-byte loads, each of which touches 32
// sectors half (a sector is requested twice, from L2 the second time).
template <int BITS, int NB, bool WIDE>
__global__ void __launch_bounds__(kLThreads)
    laaq_quantize_kernel(const uint16_t *__restrict__ x, int64_t nblocks, uint8_t *__restrict__ packed,
                         float *__restrict__ scale)
{
    constexpr int LPB = NB / 32;
    constexpr int U = kQuantSlots;
    const uint64_t pol = WIDE ? policy_evict_first() : 0;  // the input is read once
    pdl_wait();
    const int64_t total = nblocks * LPB;
    const int lane = threadIdx.x & 31;
    const int part = lane % LPB;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
         base += U * stride) {
        uint4 g[U][4];
        int64_t off[U];
        bool valid[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t t = base + u * stride + lane;
            valid[u] = t < total;
            off[u] = (valid[u] ? t / LPB : 0) * NB + part * 32;
            if constexpr (WIDE) {
                if (valid[u]) {
                    ldg256_stream_hint(x + off[u], pol, g[u][0], g[u][1]);
                    ldg256_stream_hint(x + off[u] + 16, pol, g[u][2], g[u][3]);
                } else {
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        g[u][h] = make_uint4(0, 0, 0, 0);
                }
            } else {
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    g[u][h] = valid[u] ? ldg128_stream(x + off[u] + 8 * h) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float v[32];
            float mx = 0.0f;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint32_t gw[4] = {g[u][h].x, g[u][h].y, g[u][h].z, g[u][h].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[8 * h + 2 * j] = bf16lo_to_f32(gw[j]);
                    v[8 * h + 2 * j + 1] = bf16hi_to_f32(gw[j]);
                    mx = fmaxf(mx, fmaxf(fabsf(v[8 * h + 2 * j]), fabsf(v[8 * h + 2 * j + 1])));
                }
            }
            const float amax = group_max<LPB>(mx);
            float q, m;
            laaq_factors<BITS>(amax, q, m);
            // |x q| <= qmax up to one rounding, so the clamp to +-qmax never
            // binds: the nearest integer of qmax (1 + 2^-23) is qmax
            uint32_t c[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                c[i] = __float_as_uint(__fadd_rn(__fmul_rn(v[i], q), kRoundMagic));
            uint32_t w[BITS];
            pack32<BITS>(c, w);
            if (valid[u]) {
                store_words<BITS>(packed + off[u] * BITS / 8, w);
                if (part == 0)
                    scale[off[u] / NB] = m;
            }
        }
    }
}

// The dequantizer works on warp tiles of 1024 codes (128 units of 8 codes;
// 128 * BITS bytes of the stream, 16-byte aligned).  Lane l decodes units
// l, 32 + l, 64 + l and 96 + l of its tile, so each of its four 16-byte
// bf16 stores (two fp32 ones) joins the warp's into one contiguous 512-byte
// (1 KB) run.  A unit's 8 * BITS bits are held as two 32-bit words, code 0
// in the lowest bits of lo.  At 4 and 8 bits a unit is one aligned 4- or
// 8-byte load, and a warp's loads of one unit index are contiguous.  At 5
// and 6 bits a unit is not word-aligned, so the warp loads the tile with
// 16-byte loads into its shared buffer and each lane takes its two words
// from there.  Codes become floats with the magic-number trick (one logic
// operation after the shift) and are scaled two at a time with packed
// fp32x2 instructions.
struct UnitBits {
    uint32_t lo, hi;
};

// Code i (0..7) of a unit as a float 1.5 * 2^23 + code + 2^(BITS-1): the
// BITS-bit field with its sign bit flipped is code + 2^(BITS-1) in
// [0, 2^BITS), and placed in the low mantissa bits of 1.5 * 2^23 (with
// which it shares no bit) it gives that float.  One exact subtraction of
// 1.5 * 2^23 + 2^(BITS-1) leaves the code.
template <int BITS> __device__ __forceinline__ float biased_code(const UnitBits &u, int i)
{
    constexpr uint32_t kMask = (1u << BITS) - 1u, kSign = 1u << (BITS - 1);
    const int bit = BITS * i;
    uint32_t raw;
    if (bit + BITS <= 32)
        raw = u.lo >> bit;
    else if (bit >= 32)
        raw = u.hi >> (bit - 32);
    else
        raw = __funnelshift_r(u.lo, u.hi, bit);
    return __uint_as_float((raw & kMask) ^ (kSign | 0x4B400000u));
}

constexpr int kTileUnits = 128;                  // units of 8 codes per warp tile
constexpr int kTileCodes = 8 * kTileUnits;       // 1024

// The operator applied after dequantisation: none, or SiLU recomputed from
// the stored input (AGoQ 2.A: RMSNorm and SiLU keep only their quantised
// input and recompute their output).
constexpr int kOpNone = 0, kOpSilu = 1;

// The unit's 8 values x_hat = code * m: an exact subtraction, then one
// rounded multiply (two values at a time).
template <int BITS> __device__ __forceinline__ void decode_unit(const UnitBits &u, float m, float2 (&v)[4])
{
    constexpr float kBias = kRoundMagic + static_cast<float>(1 << (BITS - 1));
    const float2 nb2 = make_float2(-kBias, -kBias), m2 = make_float2(m, m);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = __fmul2_rn(__fadd2_rn(make_float2(biased_code<BITS>(u, 2 * i), biased_code<BITS>(u, 2 * i + 1)),
                                     nb2),
                          m2);
}

// SiLU(x) = x sigma(x) in fp32, from e = exp(-|x|) <= 1 (expf, at most 2
// units in the last place; it cannot overflow): sigma(|x|) = 1 / (1 + e) and
// sigma(-|x|) = e / (1 + e).  The reciprocal of 1 + e, which lies in [1, 2],
// is __fdividef's (at most 2 units in the last place there); the result is
// then within about 6 units in the last place of x sigma(x).
__device__ __forceinline__ float silu(float x)
{
    const float e = expf(-fabsf(x));
    const float r = __fdividef(1.0f, 1.0f + e);
    return x * (x >= 0.0f ? r : e * r);
}

// Stores 8 consecutive fp32 values at element 8 unit of `out`, as fp32 or
// rounded to bf16 (nearest, ties to even).
template <bool BF16OUT> __device__ __forceinline__ void store_unit(const float2 (&v)[4], void *out, int64_t unit)
{
    if constexpr (BF16OUT) {
        stg128_stream(static_cast<uint16_t *>(out) + 8 * unit,
                      make_uint4(f32x2_to_bf16x2(v[0].x, v[0].y), f32x2_to_bf16x2(v[1].x, v[1].y),
                                 f32x2_to_bf16x2(v[2].x, v[2].y), f32x2_to_bf16x2(v[3].x, v[3].y)));
    } else {
        float *o = static_cast<float *>(out) + 8 * unit;
        stg128_stream(o, make_uint4(__float_as_uint(v[0].x), __float_as_uint(v[0].y), __float_as_uint(v[1].x),
                                    __float_as_uint(v[1].y)));
        stg128_stream(o + 4, make_uint4(__float_as_uint(v[2].x), __float_as_uint(v[2].y),
                                        __float_as_uint(v[3].x), __float_as_uint(v[3].y)));
    }
}

template <int BITS, bool BF16OUT, int OP>
__device__ __forceinline__ void decode_store_unit(const UnitBits &u, float m, void *out, int64_t unit)
{
    float2 v[4];
    decode_unit<BITS>(u, m, v);
    if constexpr (OP == kOpSilu) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = make_float2(silu(v[i].x), silu(v[i].y));
    }
    store_unit<BF16OUT>(v, out, unit);
}

template <int BITS, int NB, bool BF16OUT, int OP>
__global__ void __launch_bounds__(kLThreads)
    laaq_dequantize_kernel(const uint8_t *__restrict__ packed, const float *__restrict__ scale, int64_t n,
                           void *__restrict__ out)
{
    constexpr bool kStaged = (BITS == 5 || BITS == 6);
    constexpr int kTileBytes = kTileUnits * BITS;   // 640 or 768 at 5 / 6 bits
    constexpr int kChunks = kTileBytes / 16;        // 16-byte chunks per tile: 40 or 48
    __shared__ __align__(16) uint8_t stage[kLThreads / 32][kStaged ? kTileBytes : 16];
    pdl_wait();
    const int lane = threadIdx.x & 31;
    uint8_t *buf = stage[threadIdx.x >> 5];
    const int64_t units = n / 8;
    const int64_t nbytes = units * BITS;
    const int64_t ntiles = (units + kTileUnits - 1) / kTileUnits;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kLThreads / 32);
    for (int64_t tile = static_cast<int64_t>(blockIdx.x) * (kLThreads / 32) + (threadIdx.x >> 5); tile < ntiles;
         tile += nwarps) {
        const int64_t u0 = tile * kTileUnits;                  // first unit of the tile
        const bool full = u0 + kTileUnits <= units;            // warp-uniform
        UnitBits w[4];
        float m[4];
        if constexpr (kStaged) {
            // the tile's bytes: chunks lane and 32 + lane (the second only for
            // lanes below kChunks - 32), whole words at the stream's ragged end
            const uint8_t *src = packed + u0 * BITS;
            uint4 c0 = make_uint4(0, 0, 0, 0), c1 = make_uint4(0, 0, 0, 0);
            if (full) {
                c0 = ldg128_stream(src + 16 * lane);
                if (lane < kChunks - 32)
                    c1 = ldg128_stream(src + 16 * (32 + lane));
            } else {
                const int64_t left = nbytes - u0 * BITS;           // bytes of the tile in the stream
                uint32_t t[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int64_t off = 16 * (32 * h + lane) + 4 * k;
                        if ((h == 0 || lane < kChunks - 32) && off < left)
                            t[4 * h + k] = __ldg(reinterpret_cast<const uint32_t *>(src + off));
                    }
                c0 = make_uint4(t[0], t[1], t[2], t[3]);
                c1 = make_uint4(t[4], t[5], t[6], t[7]);
            }
            __syncwarp();  // the previous tile's words have been read
            *reinterpret_cast<uint4 *>(buf + 16 * lane) = c0;
            if (lane < kChunks - 32)
                *reinterpret_cast<uint4 *>(buf + 16 * (32 + lane)) = c1;
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int byte = BITS * (32 * k + lane), a = byte & ~3;
                const uint32_t sh = 8u * static_cast<uint32_t>(byte & 3);
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(buf + a);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(buf + a + 4);
                w[k] = {__funnelshift_r(w0, w1, sh), w1 >> sh};
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t u = u0 + 32 * k + lane;
                w[k] = {0u, 0u};
                if (full || u < units) {
                    if constexpr (BITS == 8) {
                        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(packed) + u);
                        w[k] = {v.x, v.y};
                    } else {
                        w[k] = {__ldg(reinterpret_cast<const uint32_t *>(packed) + u), 0u};
                    }
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t u = u0 + 32 * k + lane;
            m[k] = (full || u < units) ? __ldg(scale + u / (NB / 8)) : 1.0f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t u = u0 + 32 * k + lane;
            if (full || u < units)
                decode_store_unit<BITS, BF16OUT, OP>(w[k], m[k], out, u);
        }
    }
}

// RMSNorm recomputed from the stored quantised input (AGoQ 2.A): rows of d
// values (d a multiple of the block, so a row holds whole blocks), one warp
// per row and two passes over the row's values.  Pass 1: the sum of x_hat^2,
// each 8-code unit as a chain of fused multiply-adds, the units of a lane in
// a compensated (Kahan) sum, the lanes by shuffles; pass 2:
// y = x_hat * (1 / sqrt(sum / d + eps)) * g, with IEEE square root and
// division.  A lane loads all its units of a row at once and keeps the
// packed words for pass 2 (UPL units at most); longer rows re-read their
// codes in pass 2 from L1 / L2 (UPL = 0).
//
// A unit of 8 codes is BITS bytes at byte 8 BITS u / 8 of the stream: one
// aligned word (4 bits) or two (8 bits); at 5 and 6 bits it starts inside a
// word and spans at most two aligned words (the second read only while it is
// inside the stream).
template <int BITS> __device__ __forceinline__ UnitBits load_unit(const uint8_t *packed, int64_t u, int64_t nbytes)
{
    if constexpr (BITS == 4) {
        return {__ldg(reinterpret_cast<const uint32_t *>(packed) + u), 0u};
    } else if constexpr (BITS == 8) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(packed) + u);
        return {v.x, v.y};
    } else {
        const int64_t byte = u * BITS, a = byte & ~int64_t(3);
        const uint32_t sh = 8u * static_cast<uint32_t>(byte & 3);
        const uint32_t w0 = __ldg(reinterpret_cast<const uint32_t *>(packed + a));
        const uint32_t w1 = a + 4 < nbytes ? __ldg(reinterpret_cast<const uint32_t *>(packed + a + 4)) : 0u;
        return {__funnelshift_r(w0, w1, sh), w1 >> sh};
    }
}

template <int BITS, int NB, bool BF16OUT, int UPL>
__global__ void __launch_bounds__(kLThreads)
    laaq_rmsnorm_kernel(const uint8_t *__restrict__ packed, const float *__restrict__ scale, int64_t rows,
                        int64_t d, const float *__restrict__ gamma, float eps, void *__restrict__ out)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t upr = d / 8;  // units per row
    const int64_t nbytes = rows * d * BITS / 8;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (kLThreads / 32);
    const float inv_d = 1.0f / static_cast<float>(d);
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * (kLThreads / 32) + (threadIdx.x >> 5); r < rows;
         r += nwarps) {
        const int64_t u0 = r * upr;
        float sum = 0.0f, comp = 0.0f;  // Kahan: sum + comp carries the lane's total
        auto add_unit = [&](const float2 (&v)[4]) {
            float t = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                t = fmaf(v[i].x, v[i].x, t);
                t = fmaf(v[i].y, v[i].y, t);
            }
            const float yk = t - comp;
            const float tk = sum + yk;
            comp = (tk - sum) - yk;
            sum = tk;
        };
        auto store_scaled = [&](float2 (&v)[4], int64_t j, float inv) {
            const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gamma + 8 * j));
            const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gamma + 8 * j + 4));
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = make_float2(v[i].x * inv * g[2 * i], v[i].y * inv * g[2 * i + 1]);
            store_unit<BF16OUT>(v, out, u0 + j);
        };
        if constexpr (UPL > 0) {
            // the lane's units of the row (at most UPL), loaded at once and
            // kept as packed words for both passes
            UnitBits w[UPL];
            float m[UPL];
#pragma unroll
            for (int k = 0; k < UPL; ++k) {
                const int64_t j = lane + 32 * k;
                w[k] = {0u, 0u};
                m[k] = 0.0f;
                if (j < upr) {
                    w[k] = load_unit<BITS>(packed, u0 + j, nbytes);
                    m[k] = __ldg(scale + (u0 + j) / (NB / 8));
                }
            }
#pragma unroll
            for (int k = 0; k < UPL; ++k) {
                if (lane + 32 * k < upr) {
                    float2 v[4];
                    decode_unit<BITS>(w[k], m[k], v);
                    add_unit(v);
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
            const float inv = 1.0f / sqrtf(sum * inv_d + eps);
#pragma unroll
            for (int k = 0; k < UPL; ++k) {
                const int64_t j = lane + 32 * k;
                if (j < upr) {
                    float2 v[4];
                    decode_unit<BITS>(w[k], m[k], v);
                    store_scaled(v, j, inv);
                }
            }
        } else {
            // long rows: two passes over the row's codes (the second from L1 / L2)
#pragma unroll 4
            for (int64_t j = lane; j < upr; j += 32) {
                float2 v[4];
                decode_unit<BITS>(load_unit<BITS>(packed, u0 + j, nbytes), __ldg(scale + (u0 + j) / (NB / 8)), v);
                add_unit(v);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
            const float inv = 1.0f / sqrtf(sum * inv_d + eps);
#pragma unroll 4
            for (int64_t j = lane; j < upr; j += 32) {
                float2 v[4];
                decode_unit<BITS>(load_unit<BITS>(packed, u0 + j, nbytes), __ldg(scale + (u0 + j) / (NB / 8)), v);
                store_scaled(v, j, inv);
            }
        }
    }
}

template <typename K> cudaError_t laaq_grid(K kernel, int64_t lanes, int *grid)
{
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kLThreads, 0)) != cudaSuccess)
        return e;
    const int64_t need = (lanes + kLThreads - 1) / kLThreads;
    const int64_t cap = static_cast<int64_t>(di.num_sms) * (per_sm < 1 ? 1 : per_sm);
    *grid = static_cast<int>(need < cap ? need : cap);
    return cudaSuccess;
}

template <int BITS, int NB, bool WIDE>
cudaError_t run_quantize_w(const void *x, int64_t n, uint8_t *packed, float *scale, cudaStream_t st)
{
    int grid = 0;
    const int64_t nb = n / NB;
    cudaError_t e = laaq_grid(laaq_quantize_kernel<BITS, NB, WIDE>, nb * (NB / 32), &grid);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(laaq_quantize_kernel<BITS, NB, WIDE>, grid, kLThreads, 0, st,
                      static_cast<const uint16_t *>(x), nb, packed, scale);
}

template <int BITS, int NB>
cudaError_t run_quantize(const void *x, int64_t n, uint8_t *packed, float *scale, cudaStream_t st)
{
    if (reinterpret_cast<uintptr_t>(x) % 32 == 0)
        return run_quantize_w<BITS, NB, true>(x, n, packed, scale, st);
    return run_quantize_w<BITS, NB, false>(x, n, packed, scale, st);
}

template <int BITS, int NB, bool BF16OUT, int OP>
cudaError_t run_dequantize_k(const uint8_t *packed, const float *scale, int64_t n, void *out, cudaStream_t st)
{
    int grid = 0;
    const int64_t lanes = (n / 8 + kTileUnits - 1) / kTileUnits * 32;  // one warp per tile
    cudaError_t e = laaq_grid(laaq_dequantize_kernel<BITS, NB, BF16OUT, OP>, lanes, &grid);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(laaq_dequantize_kernel<BITS, NB, BF16OUT, OP>, grid, kLThreads, 0, st, packed, scale, n, out);
}

template <int BITS, int NB>
cudaError_t run_dequantize(const uint8_t *packed, const float *scale, int64_t n, void *out, bool bf16, int op,
                           cudaStream_t st)
{
    if (op == kOpSilu)
        return bf16 ? run_dequantize_k<BITS, NB, true, kOpSilu>(packed, scale, n, out, st)
                    : run_dequantize_k<BITS, NB, false, kOpSilu>(packed, scale, n, out, st);
    return bf16 ? run_dequantize_k<BITS, NB, true, kOpNone>(packed, scale, n, out, st)
                : run_dequantize_k<BITS, NB, false, kOpNone>(packed, scale, n, out, st);
}

template <int BITS>
cudaError_t quantize_nb(int block, const void *x, int64_t n, uint8_t *packed, float *scale, cudaStream_t st)
{
    switch (block) {
    case 32:
        return run_quantize<BITS, 32>(x, n, packed, scale, st);
    case 64:
        return run_quantize<BITS, 64>(x, n, packed, scale, st);
    case 128:
        return run_quantize<BITS, 128>(x, n, packed, scale, st);
    default:
        return run_quantize<BITS, 256>(x, n, packed, scale, st);
    }
}

template <int BITS>
cudaError_t dequantize_nb(int block, const uint8_t *packed, const float *scale, int64_t n, void *out, bool bf16,
                          int op, cudaStream_t st)
{
    switch (block) {
    case 32:
        return run_dequantize<BITS, 32>(packed, scale, n, out, bf16, op, st);
    case 64:
        return run_dequantize<BITS, 64>(packed, scale, n, out, bf16, op, st);
    case 128:
        return run_dequantize<BITS, 128>(packed, scale, n, out, bf16, op, st);
    default:
        return run_dequantize<BITS, 256>(packed, scale, n, out, bf16, op, st);
    }
}

}  // namespace

cudaError_t launch_laaq_quantize(const void *x_bf16, int64_t n, int block, int bits, uint8_t *packed,
                                 float *scale, cudaStream_t stream)
{
    switch (bits) {
    case 4:
        return quantize_nb<4>(block, x_bf16, n, packed, scale, stream);
    case 5:
        return quantize_nb<5>(block, x_bf16, n, packed, scale, stream);
    case 6:
        return quantize_nb<6>(block, x_bf16, n, packed, scale, stream);
    default:
        return quantize_nb<8>(block, x_bf16, n, packed, scale, stream);
    }
}

namespace {

template <int BITS, int NB, bool BF16OUT, int UPL>
cudaError_t run_rmsnorm_k(const uint8_t *packed, const float *scale, int64_t rows, int64_t d, const float *gamma,
                          float eps, void *out, cudaStream_t st)
{
    int grid = 0;
    cudaError_t e = laaq_grid(laaq_rmsnorm_kernel<BITS, NB, BF16OUT, UPL>, rows * 32, &grid);  // a warp per row
    if (e != cudaSuccess)
        return e;
    return launch_pdl(laaq_rmsnorm_kernel<BITS, NB, BF16OUT, UPL>, grid, kLThreads, 0, st, packed, scale, rows, d,
                      gamma, eps, out);
}

// Rows of up to 16 units a lane (4096 values) keep their packed words in
// registers (4 or 16 units a lane); longer rows take two passes.  Measured
// at [8192, 4096], 4 bits: 20.9 us, against 22.6 us in two passes.
template <int BITS, int NB, bool BF16OUT>
cudaError_t run_rmsnorm_b(const uint8_t *packed, const float *scale, int64_t rows, int64_t d, const float *gamma,
                          float eps, void *out, cudaStream_t st)
{
    const int64_t upl = (d / 8 + 31) / 32;
    if (upl <= 4)
        return run_rmsnorm_k<BITS, NB, BF16OUT, 4>(packed, scale, rows, d, gamma, eps, out, st);
    if (upl <= 16)
        return run_rmsnorm_k<BITS, NB, BF16OUT, 16>(packed, scale, rows, d, gamma, eps, out, st);
    return run_rmsnorm_k<BITS, NB, BF16OUT, 0>(packed, scale, rows, d, gamma, eps, out, st);
}

template <int BITS, int NB>
cudaError_t run_rmsnorm(const uint8_t *packed, const float *scale, int64_t rows, int64_t d, const float *gamma,
                        float eps, void *out, bool bf16, cudaStream_t st)
{
    return bf16 ? run_rmsnorm_b<BITS, NB, true>(packed, scale, rows, d, gamma, eps, out, st)
                : run_rmsnorm_b<BITS, NB, false>(packed, scale, rows, d, gamma, eps, out, st);
}

template <int BITS>
cudaError_t rmsnorm_nb(int block, const uint8_t *packed, const float *scale, int64_t rows, int64_t d,
                       const float *gamma, float eps, void *out, bool bf16, cudaStream_t st)
{
    switch (block) {
    case 32:
        return run_rmsnorm<BITS, 32>(packed, scale, rows, d, gamma, eps, out, bf16, st);
    case 64:
        return run_rmsnorm<BITS, 64>(packed, scale, rows, d, gamma, eps, out, bf16, st);
    case 128:
        return run_rmsnorm<BITS, 128>(packed, scale, rows, d, gamma, eps, out, bf16, st);
    default:
        return run_rmsnorm<BITS, 256>(packed, scale, rows, d, gamma, eps, out, bf16, st);
    }
}

}  // namespace

cudaError_t launch_laaq_rmsnorm(const uint8_t *packed, const float *scale, int64_t rows, int64_t d, int block,
                                int bits, const float *gamma, float eps, void *out, bool out_bf16,
                                cudaStream_t stream)
{
    switch (bits) {
    case 4:
        return rmsnorm_nb<4>(block, packed, scale, rows, d, gamma, eps, out, out_bf16, stream);
    case 5:
        return rmsnorm_nb<5>(block, packed, scale, rows, d, gamma, eps, out, out_bf16, stream);
    case 6:
        return rmsnorm_nb<6>(block, packed, scale, rows, d, gamma, eps, out, out_bf16, stream);
    default:
        return rmsnorm_nb<8>(block, packed, scale, rows, d, gamma, eps, out, out_bf16, stream);
    }
}

cudaError_t launch_laaq_dequantize(const uint8_t *packed, const float *scale, int64_t n, int block, int bits,
                                   void *out, bool out_bf16, bool silu, cudaStream_t stream)
{
    const int op = silu ? kOpSilu : kOpNone;
    switch (bits) {
    case 4:
        return dequantize_nb<4>(block, packed, scale, n, out, out_bf16, op, stream);
    case 5:
        return dequantize_nb<5>(block, packed, scale, n, out, out_bf16, op, stream);
    case 6:
        return dequantize_nb<6>(block, packed, scale, n, out, out_bf16, op, stream);
    default:
        return dequantize_nb<8>(block, packed, scale, n, out, out_bf16, op, stream);
    }
}

}  // namespace taco
