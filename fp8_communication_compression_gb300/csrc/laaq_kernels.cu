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
// A lane owns 32 consecutive elements of a block; its 32 codes are exactly
// b 32-bit words of the stream, packed with compile-time shifts.

#include <cfloat>

#include "device_utils.cuh"
#include "internal.h"
#include "reduce_math.cuh"

namespace taco {

namespace {

constexpr int kLThreads = 256;

template <int BITS> __device__ __forceinline__ void pack32(const int (&c)[32], uint32_t (&w)[BITS])
{
    constexpr uint32_t kMask = (1u << BITS) - 1u;
#pragma unroll
    for (int j = 0; j < BITS; ++j)
        w[j] = 0u;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t u = static_cast<uint32_t>(c[i]) & kMask;
        const int pos = i * BITS, wi = pos / 32, sh = pos % 32;
        w[wi] |= u << sh;
        if (sh + BITS > 32)
            w[wi + 1] |= u >> (32 - sh);
    }
}

template <int BITS> __device__ __forceinline__ int unpack_one(const uint32_t (&w)[BITS], int i)
{
    const int pos = i * BITS, wi = pos / 32, sh = pos % 32;
    uint32_t raw = w[wi] >> sh;
    if (sh + BITS > 32)
        raw |= w[wi + 1] << (32 - sh);
    return static_cast<int>(raw << (32 - BITS)) >> (32 - BITS);  // sign-extend
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

template <int BITS> __device__ __forceinline__ void load_words(const uint8_t *src, uint32_t (&w)[BITS])
{
    if constexpr (BITS % 4 == 0) {
#pragma unroll
        for (int j = 0; j < BITS; j += 4) {
            const uint4 q = ldg128_stream(src + 4 * j);
            w[j] = q.x;
            w[j + 1] = q.y;
            w[j + 2] = q.z;
            w[j + 3] = q.w;
        }
    } else if constexpr (BITS % 2 == 0) {
#pragma unroll
        for (int j = 0; j < BITS; j += 2) {
            const uint2 q = __ldg(reinterpret_cast<const uint2 *>(src + 4 * j));
            w[j] = q.x;
            w[j + 1] = q.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < BITS; ++j)
            w[j] = __ldg(reinterpret_cast<const uint32_t *>(src) + j);
    }
}

template <int BITS, int NB>
__global__ void __launch_bounds__(kLThreads)
    laaq_quantize_kernel(const uint16_t *__restrict__ x, int64_t nblocks, uint8_t *__restrict__ packed,
                         float *__restrict__ scale)
{
    constexpr int LPB = NB / 32;
    constexpr float kQmax = static_cast<float>((1 << (BITS - 1)) - 1);
    pdl_wait();
    pdl_launch_dependents();
    const int64_t total = nblocks * LPB;
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
         base += stride) {
        const int64_t t = base + lane;
        const bool valid = t < total;
        const int64_t blk = valid ? t / LPB : 0;
        const int part = lane % LPB;
        const int64_t off = blk * NB + part * 32;
        uint4 g[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                      make_uint4(0, 0, 0, 0)};
        if (valid) {
#pragma unroll
            for (int h = 0; h < 4; ++h)
                g[h] = ldg128_stream(x + off + 8 * h);
        }
        float v[32];
        float mx = 0.0f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint32_t gw[4] = {g[h].x, g[h].y, g[h].z, g[h].w};
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
        int c[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            c[i] = static_cast<int>(fminf(fmaxf(rintf(__fmul_rn(v[i], q)), -kQmax), kQmax));
        uint32_t w[BITS];
        pack32<BITS>(c, w);
        if (valid) {
            store_words<BITS>(packed + off * BITS / 8, w);
            if (part == 0)
                scale[blk] = m;
        }
    }
}

template <int BITS, int NB, bool BF16OUT>
__global__ void __launch_bounds__(kLThreads)
    laaq_dequantize_kernel(const uint8_t *__restrict__ packed, const float *__restrict__ scale,
                           int64_t nblocks, void *__restrict__ out)
{
    constexpr int LPB = NB / 32;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t total = nblocks * LPB;
    const int lane = threadIdx.x & 31;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31); base < total;
         base += stride) {
        const int64_t t = base + lane;
        if (t >= total)
            continue;
        const int64_t blk = t / LPB;
        const int part = lane % LPB;
        const int64_t off = blk * NB + part * 32;
        uint32_t w[BITS];
        load_words<BITS>(packed + off * BITS / 8, w);
        const float m = __ldg(scale + blk);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = __fmul_rn(static_cast<float>(unpack_one<BITS>(w, i)), m);
        if constexpr (BF16OUT) {
            uint16_t *o = static_cast<uint16_t *>(out) + off;
#pragma unroll
            for (int h = 0; h < 4; ++h)
                stg128_stream(o + 8 * h, make_uint4(f32x2_to_bf16x2(v[8 * h], v[8 * h + 1]),
                                                    f32x2_to_bf16x2(v[8 * h + 2], v[8 * h + 3]),
                                                    f32x2_to_bf16x2(v[8 * h + 4], v[8 * h + 5]),
                                                    f32x2_to_bf16x2(v[8 * h + 6], v[8 * h + 7])));
        } else {
            float *o = static_cast<float *>(out) + off;
#pragma unroll
            for (int h = 0; h < 8; ++h)
                stg128_stream(o + 4 * h, make_uint4(__float_as_uint(v[4 * h]), __float_as_uint(v[4 * h + 1]),
                                                    __float_as_uint(v[4 * h + 2]),
                                                    __float_as_uint(v[4 * h + 3])));
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
    const int64_t nb = n / NB;
    if (bf16) {
        cudaError_t e = laaq_grid(laaq_dequantize_kernel<BITS, NB, true>, nb * (NB / 32), &grid);
        if (e != cudaSuccess)
            return e;
        return launch_pdl(laaq_dequantize_kernel<BITS, NB, true>, grid, kLThreads, 0, st, packed, scale, nb, out);
    }
    cudaError_t e = laaq_grid(laaq_dequantize_kernel<BITS, NB, false>, nb * (NB / 32), &grid);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(laaq_dequantize_kernel<BITS, NB, false>, grid, kLThreads, 0, st, packed, scale, nb, out);
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
