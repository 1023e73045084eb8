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
// A lane owns 32 consecutive elements of a block; its 32 codes are exactly
// b 32-bit words of the stream, packed with compile-time shifts.  Each lane
// takes several grid-stride slots per loop trip and issues all of their
// loads before it processes the first.

#include <cfloat>

#include "device_utils.cuh"
#include "internal.h"
#include "reduce_math.cuh"

namespace taco {

namespace {

constexpr int kLThreads = 256;

// Rounding to an integer without a conversion instruction: for |v| < 2^22,
// the float sum v + 1.5 * 2^23 has a unit in the last place of 1, so the
// addition rounds v to the nearest integer (ties to even), and the low
// mantissa bits of the sum hold that integer in two's complement (the low 22
// bits of 1.5 * 2^23 are zero).
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23, bits 0x4B400000

// Packs the low BITS bits of each of 32 words (the rounded sums above) into
// the lane's BITS-word stream segment.
template <int BITS> __device__ __forceinline__ void pack32(const uint32_t (&c)[32], uint32_t (&w)[BITS])
{
    constexpr uint32_t kMask = (1u << BITS) - 1u;
#pragma unroll
    for (int j = 0; j < BITS; ++j)
        w[j] = 0u;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t u = c[i] & kMask;
        const int pos = i * BITS, wi = pos / 32, sh = pos % 32;
        w[wi] |= u << sh;
        if (sh + BITS > 32)
            w[wi + 1] |= u >> (32 - sh);
    }
}

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

template <int BITS, int NB>
__global__ void __launch_bounds__(kLThreads)
    laaq_quantize_kernel(const uint16_t *__restrict__ x, int64_t nblocks, uint8_t *__restrict__ packed,
                         float *__restrict__ scale)
{
    constexpr int LPB = NB / 32;
    constexpr int U = kQuantSlots;
    constexpr float kQmax = static_cast<float>((1 << (BITS - 1)) - 1);
    pdl_wait();
    pdl_launch_dependents();
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
#pragma unroll
            for (int h = 0; h < 4; ++h)
                g[u][h] = valid[u] ? ldg128_stream(x + off[u] + 8 * h) : make_uint4(0, 0, 0, 0);
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
            float q = 1.0f, m = 1.0f;
            if (amax > 0.0f) {
                q = fminf(kQmax / amax, FLT_MAX);
                m = amax / kQmax;
            }
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

// The dequantizer's unit is 8 consecutive codes (BITS bytes of the stream);
// adjacent lanes take adjacent units, so that a warp's code loads and its
// 16-byte bf16 stores are both contiguous.  A unit's 8 * BITS bits are held
// as two 32-bit words, code 0 in the lowest bits of lo.  For 4 and 8 bits a
// unit is one aligned load; for 5 and 6 bits it is not word-aligned, so the
// warp loads its 32 units' span with 16-byte loads into a shared buffer and
// each lane takes its two words from there.
struct UnitBits {
    uint32_t lo, hi;
};

template <int BITS> __device__ __forceinline__ UnitBits load_unit(const uint8_t *packed, int64_t unit)
{
    static_assert(BITS == 4 || BITS == 8, "5- and 6-bit units are loaded through the shared buffer");
    const int64_t byte = unit * BITS;
    if constexpr (BITS == 8) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(packed + byte));
        return {v.x, v.y};
    } else {
        return {__ldg(reinterpret_cast<const uint32_t *>(packed + byte)), 0u};
    }
}

// Code i (0..7) of a unit as an exact float: the BITS-bit field with its
// sign bit flipped is code + 2^(BITS-1) in [0, 2^BITS); placed in the low
// mantissa bits of 1.5 * 2^23 it gives the float 1.5 * 2^23 + code +
// 2^(BITS-1), from which one exact subtraction leaves the code.
template <int BITS> __device__ __forceinline__ float unit_code(const UnitBits &u, int i)
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
    // (raw & mask) has no bit in common with 1.5 * 2^23, so the sign flip and
    // the exponent bits go in with one exclusive or
    const float biased = __uint_as_float((raw & kMask) ^ (kSign | 0x4B400000u));
    return __fsub_rn(biased, kRoundMagic + static_cast<float>(kSign));
}

constexpr int kDequantUnits = 8;  // units per lane per loop trip, loads issued together

template <int BITS, int NB, bool BF16OUT>
__global__ void __launch_bounds__(kLThreads)
    laaq_dequantize_kernel(const uint8_t *__restrict__ packed, const float *__restrict__ scale, int64_t n,
                           void *__restrict__ out)
{
    constexpr int U = kDequantUnits;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t units = n / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    // for 5 and 6 bits the loop test is warp-uniform (the warp's first
    // unit), so that a warp's lanes stay together through the shared-buffer
    // exchange below
    constexpr bool kStaged = (BITS == 5 || BITS == 6);
    const int64_t lane_off = kStaged ? (threadIdx.x & 31) : 0;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base - lane_off < units;
         base += U * stride) {
        UnitBits w[U];
        float m[U];
        if constexpr (kStaged) {
            // a warp's 32 consecutive units are one 16-byte-aligned span of
            // 32 * BITS bytes: 2 * BITS lanes load it with one 16-byte load
            // each, through the warp's shared buffer to the lanes that need it
            constexpr int CH = 2 * BITS;             // 16-byte chunks per span
            constexpr int SPAN = 32 * BITS;          // bytes per span
            __shared__ __align__(16) uint8_t stage[kLThreads / 32][U * 32 * 6];
            uint8_t *buf = stage[threadIdx.x >> 5];
            const int lane = threadIdx.x & 31;
            const int64_t nbytes = units * BITS;
            uint4 c[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t off = (base - lane + u * stride) * BITS + 16 * lane;
                c[u] = make_uint4(0, 0, 0, 0);
                if (lane < CH && off < nbytes) {
                    if (off + 16 <= nbytes) {
                        c[u] = ldg128_stream(packed + off);
                    } else {  // the stream ends inside this chunk: whole words only
                        uint32_t t[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (off + 4 * k < nbytes)
                                t[k] = __ldg(reinterpret_cast<const uint32_t *>(packed + off + 4 * k));
                        c[u] = make_uint4(t[0], t[1], t[2], t[3]);
                    }
                }
            }
            __syncwarp();
            if (lane < CH) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    *reinterpret_cast<uint4 *>(buf + u * SPAN + 16 * lane) = c[u];
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = base + u * stride;
                const int byte = BITS * lane, a = byte & ~3;
                const uint32_t sh = 8u * static_cast<uint32_t>(byte & 3);
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(buf + u * SPAN + a);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(buf + u * SPAN + a + 4);
                w[u] = {__funnelshift_r(w0, w1, sh), w1 >> sh};
                m[u] = j < units ? __ldg(scale + j * 8 / NB) : 1.0f;
            }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t j = base + u * stride;
                w[u] = {0u, 0u};
                m[u] = 1.0f;
                if (j < units) {
                    w[u] = load_unit<BITS>(packed, j);
                    m[u] = __ldg(scale + j * 8 / NB);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t j = base + u * stride;
            if (j >= units)
                break;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = __fmul_rn(unit_code<BITS>(w[u], i), m[u]);
            if constexpr (BF16OUT) {
                stg128_stream(static_cast<uint16_t *>(out) + 8 * j,
                              make_uint4(f32x2_to_bf16x2(v[0], v[1]), f32x2_to_bf16x2(v[2], v[3]),
                                         f32x2_to_bf16x2(v[4], v[5]), f32x2_to_bf16x2(v[6], v[7])));
            } else {
                float *o = static_cast<float *>(out) + 8 * j;
                stg128_stream(o, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                                            __float_as_uint(v[3])));
                stg128_stream(o + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]),
                                                __float_as_uint(v[6]), __float_as_uint(v[7])));
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

template <int BITS, int NB>
cudaError_t run_quantize(const void *x, int64_t n, uint8_t *packed, float *scale, cudaStream_t st)
{
    int grid = 0;
    const int64_t nb = n / NB;
    cudaError_t e = laaq_grid(laaq_quantize_kernel<BITS, NB>, nb * (NB / 32), &grid);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(laaq_quantize_kernel<BITS, NB>, grid, kLThreads, 0, st, static_cast<const uint16_t *>(x),
                      nb, packed, scale);
}

template <int BITS, int NB>
cudaError_t run_dequantize(const uint8_t *packed, const float *scale, int64_t n, void *out, bool bf16,
                           cudaStream_t st)
{
    int grid = 0;
    const int64_t lanes = (n / 8 + kDequantUnits - 1) / kDequantUnits;
    if (bf16) {
        cudaError_t e = laaq_grid(laaq_dequantize_kernel<BITS, NB, true>, lanes, &grid);
        if (e != cudaSuccess)
            return e;
        return launch_pdl(laaq_dequantize_kernel<BITS, NB, true>, grid, kLThreads, 0, st, packed, scale, n, out);
    }
    cudaError_t e = laaq_grid(laaq_dequantize_kernel<BITS, NB, false>, lanes, &grid);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(laaq_dequantize_kernel<BITS, NB, false>, grid, kLThreads, 0, st, packed, scale, n, out);
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
                          cudaStream_t st)
{
    switch (block) {
    case 32:
        return run_dequantize<BITS, 32>(packed, scale, n, out, bf16, st);
    case 64:
        return run_dequantize<BITS, 64>(packed, scale, n, out, bf16, st);
    case 128:
        return run_dequantize<BITS, 128>(packed, scale, n, out, bf16, st);
    default:
        return run_dequantize<BITS, 256>(packed, scale, n, out, bf16, st);
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

cudaError_t launch_laaq_dequantize(const uint8_t *packed, const float *scale, int64_t n, int block, int bits,
                                   void *out, bool out_bf16, cudaStream_t stream)
{
    switch (bits) {
    case 4:
        return dequantize_nb<4>(block, packed, scale, n, out, out_bf16, stream);
    case 5:
        return dequantize_nb<5>(block, packed, scale, n, out, out_bf16, stream);
    case 6:
        return dequantize_nb<6>(block, packed, scale, n, out, out_bf16, stream);
    default:
        return dequantize_nb<8>(block, packed, scale, n, out, out_bf16, stream);
    }
}

}  // namespace taco
