// C ABI of the library (include/taco.h): argument validation on the host,
// then one kernel launch on the caller's stream.  No allocation, no
// synchronisation, no exception crosses this boundary.  The host pipeline
// calls are the exception their declarations state: a pipeline owns CUDA
// streams and events, and one run enqueues copies and launches per chunk.

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <new>

#include "../../include/taco.h"
#include "internal.h"

namespace taco {

cudaError_t current_device_info(DeviceInfo *out)
{
    constexpr int kMax = 64;
    static DeviceInfo cache[kMax];
    static bool ready[kMax];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMax)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
        DeviceInfo di{dev, 0, 0};
        if ((e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
            return e;
        cache[dev] = di;
        ready[dev] = true;
    }
    *out = cache[dev];
    return cudaSuccess;
}

}  // namespace taco

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// [a, a + na) and [b, b + nb) overlap
bool overlap(const void *a, uint64_t na, const void *b, uint64_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na && nb && x < y + nb && y < x + na;
}

bool positive_finite(float v) { return std::isfinite(v) && v > 0.0f; }

taco_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TACO_OK : TACO_ERR_CUDA; }

// The 128-element row view used by the TMA kernels must fit int32 tile
// coordinates.
constexpr int64_t kMaxRows128 = (int64_t(1) << 31) - 256;

taco_status check_taco_shape(int64_t rows, int64_t d, int32_t block)
{
    if (rows < 0 || d <= 0)
        return TACO_ERR_INVALID_ARG;
    if (!taco_block_supported(block))
        return TACO_ERR_UNSUPPORTED;
    if (d % block != 0)
        return TACO_ERR_INVALID_ARG;
    if (rows > 0 && d > INT64_MAX / rows)
        return TACO_ERR_INVALID_ARG;
    if (rows * d / 128 > kMaxRows128)
        return TACO_ERR_UNSUPPORTED;
    return TACO_OK;
}


// Shared checks of the two reduce entry points; fills `sp`.  `out` (the
// optional reconstruction of the sum) may be null.
taco_status check_reduce_args(int32_t P, const uint8_t *const *codes, const float *const *alpha,
                                     const float *const *scale, int64_t rows, int64_t d, int32_t block,
                                     float e_target, float eps, const uint8_t *out_codes,
                                     const float *out_alpha, const float *out_scale, const void *out,
                                     uint64_t out_bytes_per_elem, taco::ShardPtrs *sp)
{
    taco_status st = check_taco_shape(rows, d, block);
    if (st != TACO_OK)
        return st;
    if (P < 1 || P > TACO_MAX_SHARDS)
        return TACO_ERR_UNSUPPORTED;
    if (!positive_finite(e_target) || !positive_finite(eps))
        return TACO_ERR_INVALID_ARG;
    if (rows == 0)
        return TACO_OK;
    if (!codes || !alpha || !scale || !out_codes || !out_alpha || !out_scale)
        return TACO_ERR_INVALID_ARG;
    const uint64_t n = static_cast<uint64_t>(rows * d), nb = n / block;
    if (!aligned(out_codes, 16) || !aligned(out_alpha, 4) || !aligned(out_scale, 4) ||
        (out && !aligned(out, 16)))
        return TACO_ERR_MISALIGNED;
    const void *outs[4] = {out_codes, out_alpha, out_scale, out};
    const uint64_t olen[4] = {n, 4 * nb, 4 * nb, out ? n * out_bytes_per_elem : 0};
    for (int i = 0; i < 4; ++i)
        for (int j = i + 1; j < 4; ++j)
            if (overlap(outs[i], olen[i], outs[j], olen[j]))
                return TACO_ERR_INVALID_ARG;
    for (int p = 0; p < P; ++p) {
        if (!codes[p] || !alpha[p] || !scale[p])
            return TACO_ERR_INVALID_ARG;
        if (!aligned(codes[p], 16) || !aligned(alpha[p], 4) || !aligned(scale[p], 4))
            return TACO_ERR_MISALIGNED;
        const void *ins[3] = {codes[p], alpha[p], scale[p]};
        const uint64_t lens[3] = {n, 4 * nb, 4 * nb};
        for (int i = 0; i < 3; ++i)
            for (int j = 0; j < 4; ++j)
                if (overlap(ins[i], lens[i], outs[j], olen[j]))
                    return TACO_ERR_INVALID_ARG;
        sp->codes[p] = codes[p];
        sp->alpha[p] = alpha[p];
        sp->scale[p] = scale[p];
    }
    return TACO_OK;
}

}  // namespace

extern "C" {

const char *taco_status_string(taco_status s)
{
    switch (s) {
    case TACO_OK:
        return "ok";
    case TACO_ERR_INVALID_ARG:
        return "invalid argument";
    case TACO_ERR_UNSUPPORTED:
        return "unsupported block size, shard count or size";
    case TACO_ERR_MISALIGNED:
        return "misaligned pointer";
    case TACO_ERR_CUDA:
        return "CUDA error";
    }
    return "unknown status";
}

int taco_abi_version(void) { return TACO_ABI_VERSION; }

int taco_block_supported(int32_t block) { return block == 128 || block == 256; }

static taco_status compress_any(const void *x_bf16, int64_t rows, int64_t d, int32_t block, float e_target,
                                float eps, uint8_t *codes, float *alpha, float *scale, bool int8_codes,
                                taco_stream_t stream)
{
    taco_status st = check_taco_shape(rows, d, block);
    if (st != TACO_OK)
        return st;
    if (!positive_finite(e_target) || !positive_finite(eps))
        return TACO_ERR_INVALID_ARG;
    if (rows == 0)
        return TACO_OK;
    if (!x_bf16 || !codes || !alpha || !scale)
        return TACO_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(codes, 16) || !aligned(alpha, 4) || !aligned(scale, 4))
        return TACO_ERR_MISALIGNED;
    const uint64_t n = static_cast<uint64_t>(rows * d), nb = n / block;
    if (overlap(x_bf16, 2 * n, codes, n) || overlap(x_bf16, 2 * n, alpha, 4 * nb) ||
        overlap(x_bf16, 2 * n, scale, 4 * nb) || overlap(codes, n, alpha, 4 * nb) ||
        overlap(codes, n, scale, 4 * nb) || overlap(alpha, 4 * nb, scale, 4 * nb))
        return TACO_ERR_INVALID_ARG;
    return from_cuda(taco::launch_compress(x_bf16, rows * d / 128, block, e_target, eps, codes, alpha,
                                           scale, int8_codes, reinterpret_cast<cudaStream_t>(stream)));
}

taco_status taco_compress(const void *x_bf16, int64_t rows, int64_t d, int32_t block, float e_target,
                          float eps, uint8_t *codes, float *alpha, float *scale, taco_stream_t stream)
{
    return compress_any(x_bf16, rows, d, block, e_target, eps, codes, alpha, scale, false, stream);
}

taco_status taco_compress_int8(const void *x_bf16, int64_t rows, int64_t d, int32_t block, float e_target,
                               float eps, int8_t *codes, float *alpha, float *scale, taco_stream_t stream)
{
    return compress_any(x_bf16, rows, d, block, e_target, eps, reinterpret_cast<uint8_t *>(codes), alpha,
                        scale, true, stream);
}

static taco_status decompress_any(const uint8_t *codes, const float *alpha, const float *scale, int64_t rows,
                                  int64_t d, int32_t block, void *out, int32_t out_is_bf16, bool int8_codes,
                                  taco_stream_t stream)
{
    taco_status st = check_taco_shape(rows, d, block);
    if (st != TACO_OK)
        return st;
    if (rows == 0)
        return TACO_OK;
    if (!codes || !alpha || !scale || !out)
        return TACO_ERR_INVALID_ARG;
    if (!aligned(codes, 16) || !aligned(out, 16) || !aligned(alpha, 4) || !aligned(scale, 4))
        return TACO_ERR_MISALIGNED;
    const uint64_t n = static_cast<uint64_t>(rows * d), nb = n / block;
    const uint64_t out_bytes = n * (out_is_bf16 ? 2 : 4);
    if (overlap(out, out_bytes, codes, n) || overlap(out, out_bytes, alpha, 4 * nb) ||
        overlap(out, out_bytes, scale, 4 * nb))
        return TACO_ERR_INVALID_ARG;
    return from_cuda(taco::launch_decompress(codes, alpha, scale, rows * d / 128, block, out,
                                             out_is_bf16 != 0, int8_codes,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

taco_status taco_decompress(const uint8_t *codes, const float *alpha, const float *scale, int64_t rows,
                            int64_t d, int32_t block, void *out, int32_t out_is_bf16,
                            taco_stream_t stream)
{
    return decompress_any(codes, alpha, scale, rows, d, block, out, out_is_bf16, false, stream);
}

taco_status taco_decompress_int8(const int8_t *codes, const float *alpha, const float *scale, int64_t rows,
                                 int64_t d, int32_t block, void *out, int32_t out_is_bf16,
                                 taco_stream_t stream)
{
    return decompress_any(reinterpret_cast<const uint8_t *>(codes), alpha, scale, rows, d, block, out,
                          out_is_bf16, true, stream);
}

taco_status taco_reduce_shards(int32_t P, const uint8_t *const *codes, const float *const *alpha,
                               const float *const *scale, int64_t rows, int64_t d, int32_t block,
                               float e_target, float eps, uint8_t *out_codes, float *out_alpha,
                               float *out_scale, taco_stream_t stream)
{
    taco::ShardPtrs sp{};
    taco_status st = check_reduce_args(P, codes, alpha, scale, rows, d, block, e_target, eps, out_codes,
                                       out_alpha, out_scale, nullptr, 0, &sp);
    if (st != TACO_OK || rows == 0)
        return st;
    return from_cuda(taco::launch_taco_reduce(P, sp, rows * d / block, block, e_target, eps, out_codes,
                                              out_alpha, out_scale, reinterpret_cast<cudaStream_t>(stream)));
}

taco_status taco_reduce_decompress(int32_t P, const uint8_t *const *codes, const float *const *alpha,
                                   const float *const *scale, int64_t rows, int64_t d, int32_t block,
                                   float e_target, float eps, uint8_t *out_codes, float *out_alpha,
                                   float *out_scale, void *out, int32_t out_is_bf16, taco_stream_t stream)
{
    taco::ShardPtrs sp{};
    if (rows > 0 && !out)
        return TACO_ERR_INVALID_ARG;
    taco_status st = check_reduce_args(P, codes, alpha, scale, rows, d, block, e_target, eps, out_codes,
                                       out_alpha, out_scale, out, out_is_bf16 ? 2 : 4, &sp);
    if (st != TACO_OK || rows == 0)
        return st;
    return from_cuda(taco::launch_reduce_decompress(P, sp, rows * d / 128, block, e_target, eps, out_codes,
                                                    out_alpha, out_scale, out, out_is_bf16 != 0,
                                                    reinterpret_cast<cudaStream_t>(stream)));
}

taco_status agoq_fp8_accumulate(uint8_t *main_codes, float *main_scale, const void *grad_bf16, int64_t n,
                                int32_t block, taco_stream_t stream)
{
    if (n < 0)
        return TACO_ERR_INVALID_ARG;
    if (!taco_block_supported(block))
        return TACO_ERR_UNSUPPORTED;
    if (n % block != 0)
        return TACO_ERR_INVALID_ARG;
    if (n == 0)
        return TACO_OK;
    if (!main_codes || !main_scale || !grad_bf16)
        return TACO_ERR_INVALID_ARG;
    if (!aligned(main_codes, 16) || !aligned(grad_bf16, 16) || !aligned(main_scale, 4))
        return TACO_ERR_MISALIGNED;
    const uint64_t nb = static_cast<uint64_t>(n / block);
    if (overlap(main_codes, n, main_scale, 4 * nb) || overlap(grad_bf16, 2 * n, main_codes, n) ||
        overlap(grad_bf16, 2 * n, main_scale, 4 * nb))
        return TACO_ERR_INVALID_ARG;
    return from_cuda(taco::launch_agoq_accumulate(main_codes, main_scale, grad_bf16, n, block,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

taco_status agoq_reduce_shards(int32_t P, const uint8_t *const *codes, const float *const *scale, int64_t n,
                               int32_t block, uint8_t *out_codes, float *out_scale, taco_stream_t stream)
{
    if (n < 0)
        return TACO_ERR_INVALID_ARG;
    if (!taco_block_supported(block) || P < 1 || P > TACO_MAX_SHARDS)
        return TACO_ERR_UNSUPPORTED;
    if (n % block != 0)
        return TACO_ERR_INVALID_ARG;
    if (n == 0)
        return TACO_OK;
    if (!codes || !scale || !out_codes || !out_scale)
        return TACO_ERR_INVALID_ARG;
    if (!aligned(out_codes, 16) || !aligned(out_scale, 4))
        return TACO_ERR_MISALIGNED;
    const uint64_t nb = static_cast<uint64_t>(n / block);
    if (overlap(out_codes, n, out_scale, 4 * nb))
        return TACO_ERR_INVALID_ARG;
    taco::ShardPtrs sp{};
    for (int p = 0; p < P; ++p) {
        if (!codes[p] || !scale[p])
            return TACO_ERR_INVALID_ARG;
        if (!aligned(codes[p], 16) || !aligned(scale[p], 4))
            return TACO_ERR_MISALIGNED;
        if (overlap(codes[p], n, out_codes, n) || overlap(codes[p], n, out_scale, 4 * nb) ||
            overlap(scale[p], 4 * nb, out_codes, n) || overlap(scale[p], 4 * nb, out_scale, 4 * nb))
            return TACO_ERR_INVALID_ARG;
        sp.codes[p] = codes[p];
        sp.scale[p] = scale[p];
    }
    return from_cuda(taco::launch_agoq_reduce(P, sp, n, block, out_codes, out_scale,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

static taco_status check_laaq(int64_t n, int32_t block, int32_t bits)
{
    if (n < 0)
        return TACO_ERR_INVALID_ARG;
    if (!(block == 32 || block == 64 || block == 128 || block == 256) ||
        !(bits == 4 || bits == 5 || bits == 6 || bits == 8))
        return TACO_ERR_UNSUPPORTED;
    if (n % block != 0)
        return TACO_ERR_INVALID_ARG;
    return TACO_OK;
}

taco_status agoq_laaq_quantize(const void *x_bf16, int64_t n, int32_t block, int32_t bits, uint8_t *packed,
                               float *scale, taco_stream_t stream)
{
    taco_status st = check_laaq(n, block, bits);
    if (st != TACO_OK || n == 0)
        return st;
    if (!x_bf16 || !packed || !scale)
        return TACO_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(packed, 16) || !aligned(scale, 4))
        return TACO_ERR_MISALIGNED;
    const uint64_t nb = static_cast<uint64_t>(n / block), pb = static_cast<uint64_t>(n) * bits / 8;
    if (overlap(x_bf16, 2 * n, packed, pb) || overlap(x_bf16, 2 * n, scale, 4 * nb) ||
        overlap(packed, pb, scale, 4 * nb))
        return TACO_ERR_INVALID_ARG;
    return from_cuda(taco::launch_laaq_quantize(x_bf16, n, block, bits, packed, scale,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

// Shared checks of the dequantizing entry points: the stream, its
// multipliers and an output of n fp32 or bf16 values that overlaps neither.
static taco_status check_laaq_out(const uint8_t *packed, const float *scale, int64_t n, int32_t block,
                                  int32_t bits, const void *out, int32_t out_is_bf16)
{
    if (!packed || !scale || !out)
        return TACO_ERR_INVALID_ARG;
    if (!aligned(packed, 16) || !aligned(scale, 4) || !aligned(out, 16))
        return TACO_ERR_MISALIGNED;
    const uint64_t nb = static_cast<uint64_t>(n / block), pb = static_cast<uint64_t>(n) * bits / 8;
    const uint64_t ob = static_cast<uint64_t>(n) * (out_is_bf16 ? 2 : 4);
    if (overlap(out, ob, packed, pb) || overlap(out, ob, scale, 4 * nb))
        return TACO_ERR_INVALID_ARG;
    return TACO_OK;
}

taco_status agoq_laaq_dequantize(const uint8_t *packed, const float *scale, int64_t n, int32_t block,
                                 int32_t bits, void *out, int32_t out_is_bf16, taco_stream_t stream)
{
    taco_status st = check_laaq(n, block, bits);
    if (st != TACO_OK || n == 0)
        return st;
    if ((st = check_laaq_out(packed, scale, n, block, bits, out, out_is_bf16)) != TACO_OK)
        return st;
    return from_cuda(taco::launch_laaq_dequantize(packed, scale, n, block, bits, out, out_is_bf16 != 0, false,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

taco_status agoq_laaq_dequantize_silu(const uint8_t *packed, const float *scale, int64_t n, int32_t block,
                                      int32_t bits, void *out, int32_t out_is_bf16, taco_stream_t stream)
{
    taco_status st = check_laaq(n, block, bits);
    if (st != TACO_OK || n == 0)
        return st;
    if ((st = check_laaq_out(packed, scale, n, block, bits, out, out_is_bf16)) != TACO_OK)
        return st;
    return from_cuda(taco::launch_laaq_dequantize(packed, scale, n, block, bits, out, out_is_bf16 != 0, true,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

taco_status agoq_laaq_dequantize_rmsnorm(const uint8_t *packed, const float *scale, int64_t rows, int64_t d,
                                         int32_t block, int32_t bits, const float *gamma, float eps, void *out,
                                         int32_t out_is_bf16, taco_stream_t stream)
{
    if (rows < 0 || d < 0 || !(eps >= 0.0f) || !(eps <= FLT_MAX))
        return TACO_ERR_INVALID_ARG;
    if (d > (int64_t(1) << 31) || (d > 0 && rows > INT64_MAX / 8 / d))
        return TACO_ERR_UNSUPPORTED;
    const int64_t n = rows * d;
    taco_status st = check_laaq(n, block, bits);
    if (st != TACO_OK)
        return st;
    if (rows == 0 || d == 0)
        return TACO_OK;
    if (d % block != 0)
        return TACO_ERR_INVALID_ARG;
    if ((st = check_laaq_out(packed, scale, n, block, bits, out, out_is_bf16)) != TACO_OK)
        return st;
    if (!gamma)
        return TACO_ERR_INVALID_ARG;
    if (!aligned(gamma, 16))
        return TACO_ERR_MISALIGNED;
    if (overlap(out, static_cast<uint64_t>(n) * (out_is_bf16 ? 2 : 4), gamma, 4 * static_cast<uint64_t>(d)))
        return TACO_ERR_INVALID_ARG;
    return from_cuda(taco::launch_laaq_rmsnorm(packed, scale, rows, d, block, bits, gamma, eps, out, out_is_bf16 != 0,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

// The GEMM shapes the tensor-core kernel takes (M, N > 0).
static bool gemm_shape_supported(int64_t M, int64_t N, int64_t K)
{
    return K > 0 && M % 128 == 0 && N % 128 == 0 && K % 64 == 0 && M / 128 <= 65535 && N <= (int64_t(1) << 30) &&
           K <= (int64_t(1) << 30) && (M / 128) * (N / 128) <= (int64_t(1) << 30);
}

// Shared checks of the GEMM entry points.  codes hold code_bits bits per
// element of Y; alpha may be null (only the compressor has one); y_out may
// be null; a null workspace or one of 0 bytes is none.
static taco_status check_gemm_args(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                   int32_t block, const uint8_t *codes, int code_bits, const float *alpha,
                                   bool need_alpha, const float *scale, const float *y_out, const void *workspace,
                                   uint64_t workspace_bytes)
{
    if (M < 0 || N < 0 || K < 0)
        return TACO_ERR_INVALID_ARG;
    if (block != 128)
        return TACO_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return TACO_OK;
    if (!gemm_shape_supported(M, N, K))
        return TACO_ERR_UNSUPPORTED;
    if (!a_bf16 || !b_bf16 || !codes || (need_alpha && !alpha) || !scale)
        return TACO_ERR_INVALID_ARG;
    const bool ws = workspace && workspace_bytes > 0;
    if (!aligned(a_bf16, 16) || !aligned(b_bf16, 16) || !aligned(codes, 16) || (alpha && !aligned(alpha, 4)) ||
        !aligned(scale, 4) || (y_out && !aligned(y_out, 16)) || (ws && !aligned(workspace, 256)))
        return TACO_ERR_MISALIGNED;
    const uint64_t mn = static_cast<uint64_t>(M) * N, nb = mn / 128;
    const void *outs[5] = {codes, alpha, scale, y_out, ws ? workspace : nullptr};
    const uint64_t olen[5] = {mn * code_bits / 8, alpha ? 4 * nb : 0, 4 * nb, y_out ? 4 * mn : 0,
                              ws ? workspace_bytes : 0};
    const void *ins[2] = {a_bf16, b_bf16};
    const uint64_t ilen[2] = {2 * static_cast<uint64_t>(M) * K, 2 * static_cast<uint64_t>(N) * K};
    for (int i = 0; i < 5; ++i) {
        for (int j = i + 1; j < 5; ++j)
            if (overlap(outs[i], olen[i], outs[j], olen[j]))
                return TACO_ERR_INVALID_ARG;
        for (int j = 0; j < 2; ++j)
            if (overlap(outs[i], olen[i], ins[j], ilen[j]))
                return TACO_ERR_INVALID_ARG;
    }
    return TACO_OK;
}

taco_status taco_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, uint64_t *bytes)
{
    if (!bytes || M < 0 || N < 0 || K < 0)
        return TACO_ERR_INVALID_ARG;
    *bytes = 0;
    if (M == 0 || N == 0)
        return TACO_OK;
    if (!gemm_shape_supported(M, N, K))
        return TACO_ERR_UNSUPPORTED;
    return from_cuda(taco::gemm_workspace_bytes(M, N, K, bytes));
}

taco_status taco_gemm_compress(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                               int32_t block, float e_target, float eps, uint8_t *codes, float *alpha,
                               float *scale, float *y_out, void *workspace, uint64_t workspace_bytes,
                               taco_stream_t stream)
{
    if (!positive_finite(e_target) || !positive_finite(eps))
        return TACO_ERR_INVALID_ARG;
    taco_status st = check_gemm_args(a_bf16, b_bf16, M, N, K, block, codes, 8, alpha, true, scale, y_out,
                                     workspace, workspace_bytes);
    if (st != TACO_OK || M == 0 || N == 0)
        return st;
    return from_cuda(taco::launch_gemm_compress(a_bf16, b_bf16, M, N, K, e_target, eps, codes, alpha, scale, y_out,
                                                workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

taco_status agoq_gemm_accumulate(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                 int32_t block, uint8_t *main_codes, float *main_scale, float *y_out,
                                 void *workspace, uint64_t workspace_bytes, taco_stream_t stream)
{
    taco_status st = check_gemm_args(a_bf16, b_bf16, M, N, K, block, main_codes, 8, nullptr, false, main_scale,
                                     y_out, workspace, workspace_bytes);
    if (st != TACO_OK || M == 0 || N == 0)
        return st;
    return from_cuda(taco::launch_gemm_agoq_accumulate(a_bf16, b_bf16, M, N, K, main_codes, main_scale, y_out,
                                                       workspace, workspace_bytes,
                                                       reinterpret_cast<cudaStream_t>(stream)));
}

taco_status agoq_gemm_laaq_quantize(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                    int32_t block, int32_t bits, uint8_t *packed, float *scale, float *y_out,
                                    void *workspace, uint64_t workspace_bytes, taco_stream_t stream)
{
    if (bits != 4 && bits != 5 && bits != 6 && bits != 8)
        return TACO_ERR_UNSUPPORTED;
    taco_status st = check_gemm_args(a_bf16, b_bf16, M, N, K, block, packed, bits, nullptr, false, scale, y_out,
                                     workspace, workspace_bytes);
    if (st != TACO_OK || M == 0 || N == 0)
        return st;
    return from_cuda(taco::launch_gemm_laaq_quantize(a_bf16, b_bf16, M, N, K, bits, packed, scale, y_out, workspace,
                                                     workspace_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

taco_status taco_e4m3_encode(const float *x, int64_t n, uint8_t *codes, taco_stream_t stream)
{
    if (n < 0)
        return TACO_ERR_INVALID_ARG;
    if (n == 0)
        return TACO_OK;
    if (!x || !codes)
        return TACO_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(codes, 16))
        return TACO_ERR_MISALIGNED;
    if (overlap(x, 4 * static_cast<uint64_t>(n), codes, static_cast<uint64_t>(n)))
        return TACO_ERR_INVALID_ARG;
    return from_cuda(taco::launch_e4m3_encode(x, n, codes, reinterpret_cast<cudaStream_t>(stream)));
}

struct taco_host_pipeline {
    taco::HostPipeline *impl;
};

taco_status taco_host_pipeline_create(int32_t P, int64_t rows, int64_t d, int32_t block, int32_t chunks,
                                      int32_t out_is_bf16, taco_host_pipeline **pipe_out,
                                      uint64_t *workspace_bytes)
{
    if (!pipe_out || !workspace_bytes)
        return TACO_ERR_INVALID_ARG;
    *pipe_out = nullptr;
    taco_status st = check_taco_shape(rows, d, block);
    if (st != TACO_OK)
        return st;
    if (P < 1 || P > TACO_MAX_SHARDS)
        return TACO_ERR_UNSUPPORTED;
    if (rows < 1 || chunks < 1 || chunks > taco::host_pipeline_max_chunks())
        return TACO_ERR_INVALID_ARG;
    auto *h = new (std::nothrow) taco_host_pipeline{nullptr};
    if (!h)
        return TACO_ERR_CUDA;
    const int c = static_cast<int>(chunks < rows ? chunks : rows);
    cudaError_t e = taco::host_pipeline_create(P, rows, d, block, c, out_is_bf16 != 0, &h->impl, workspace_bytes);
    if (e != cudaSuccess) {
        delete h;
        return TACO_ERR_CUDA;
    }
    *pipe_out = h;
    return TACO_OK;
}

taco_status taco_host_pipeline_run(taco_host_pipeline *pipe, const void *x_host_bf16, void *out_host,
                                   void *workspace, float e_target, float eps, taco_stream_t stream)
{
    if (!pipe || !pipe->impl || !x_host_bf16 || !out_host || !workspace)
        return TACO_ERR_INVALID_ARG;
    if (!positive_finite(e_target) || !positive_finite(eps))
        return TACO_ERR_INVALID_ARG;
    if (!aligned(workspace, 256))
        return TACO_ERR_MISALIGNED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return TACO_ERR_CUDA;
    if (dev != taco::host_pipeline_device(pipe->impl))
        return TACO_ERR_INVALID_ARG;
    return from_cuda(taco::host_pipeline_run(pipe->impl, x_host_bf16, out_host, workspace, e_target, eps,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

taco_status taco_host_pipeline_destroy(taco_host_pipeline *pipe)
{
    if (!pipe)
        return TACO_ERR_INVALID_ARG;
    taco::host_pipeline_destroy(pipe->impl);
    delete pipe;
    return TACO_OK;
}

taco_status taco_watchdog_selftest(taco_stream_t stream)
{
    return from_cuda(taco::launch_watchdog_selftest(reinterpret_cast<cudaStream_t>(stream)));
}

taco_status taco_device_error(uint32_t *flags_out, int32_t clear)
{
    if (!flags_out)
        return TACO_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return TACO_ERR_CUDA;
    uint32_t codec = 0, gemm = 0;
    if ((e = taco::read_codec_error(&codec, clear != 0)) != cudaSuccess ||
        (e = taco::read_gemm_error(&gemm, clear != 0)) != cudaSuccess)
        return from_cuda(e);
    *flags_out = codec | gemm;
    return TACO_OK;
}

}  // extern "C"
