// taco_two_shot_host_noalloc: the host-buffer two-shot local path for
// callers that cannot allocate device memory.
//
// taco_host_pipeline_run needs a device workspace that the caller
// allocates.  Some callers cannot: code that runs where an allocation may
// not happen (inside a memory-pool or allocator hook, a signal-safe or
// real-time section), or a host program that links this library but not an
// allocator it is allowed to use.  This entry point needs no workspace and
// allocates nothing: its intermediate buffers (the gathered bf16 shards,
// their codes and scales, the reduced codes and scales, the fp32 result)
// live in one file-scope device array, kScratchBytes long, which every GPU
// that loads the library holds until the process exits.  The rows are
// processed in chunks that fit the array, one chunk after another on the
// caller's stream: copy in, compress, reduce, decompress, copy out.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  Nothing in it needs to start at zero: each chunk writes every
// byte it later reads.  Calls whose work overlaps on the GPU (on different
// streams, or from different host threads) race on the array.
//
// Host code cannot use the array's name as a device address (in host code
// it names a host-side stand-in), so the first call on each device looks up
// the device address with cudaGetSymbolAddress and keeps it.

#include <cfloat>
#include <cstdint>
#include <mutex>

#include "../../include/taco.h"
#include "internal.h"

namespace {

constexpr uint64_t kScratchBytes = static_cast<uint64_t>(TACO_NOALLOC_SCRATCH_MIB) << 20;
constexpr uint64_t kAlign = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

uint64_t round_up(uint64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Device address of the scratch array on device `dev`, which must be the
// current device (looked up once per device).
cudaError_t scratch_address(int dev, uint8_t **out)
{
    static uint8_t *addr[kMaxDevices];
    static std::mutex mu;
    cudaError_t e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return e;
        addr[dev] = static_cast<uint8_t *>(p);
    }
    *out = addr[dev];
    return cudaSuccess;
}

// Byte offsets of one chunk's buffers in the array, for a chunk of R rows.
struct ChunkLayout {
    uint64_t x, codes, alpha, scale, rcodes, ralpha, rscale, out, total;
};

ChunkLayout layout(int P, int64_t R, int64_t d, int block)
{
    const uint64_t e = static_cast<uint64_t>(R) * d, nb = e / block;
    ChunkLayout L{};
    uint64_t off = 0;
    auto take = [&](uint64_t bytes) {
        const uint64_t o = off;
        off = round_up(off + bytes);
        return o;
    };
    L.x = take(2 * P * e);
    L.codes = take(P * e);
    L.alpha = take(4 * P * nb);
    L.scale = take(4 * P * nb);
    L.rcodes = take(e);
    L.ralpha = take(4 * nb);
    L.rscale = take(4 * nb);
    L.out = take(4 * e);
    L.total = off;
    return L;
}

// Rows per chunk: the most that fit the array (0 if one row does not).
int64_t chunk_rows(int P, int64_t rows, int64_t d, int block)
{
    const uint64_t per_row = layout(P, 1, d, block).total;
    int64_t R = static_cast<int64_t>(kScratchBytes / (per_row ? per_row : 1));
    if (R > rows)
        R = rows;
    while (R > 0 && layout(P, R, d, block).total > kScratchBytes)
        --R;
    return R;
}

}  // namespace

extern "C" {

taco_status taco_two_shot_host_noalloc(int32_t P, int64_t rows, int64_t d, int32_t block, const void *x_host_bf16,
                                       float *out_host, float e_target, float eps, taco_stream_t stream)
{
    if (!(block == 128 || block == 256) || P < 1 || P > TACO_MAX_SHARDS)
        return TACO_ERR_UNSUPPORTED;
    if (rows < 0 || d <= 0 || d % block != 0 || !(e_target > 0.0f && e_target <= FLT_MAX) ||
        !(eps > 0.0f && eps <= FLT_MAX))
        return TACO_ERR_INVALID_ARG;
    if (rows == 0)
        return TACO_OK;
    if (!x_host_bf16 || !out_host)
        return TACO_ERR_INVALID_ARG;
    const int64_t R = chunk_rows(P, rows, d, block);
    if (R < 1)
        return TACO_ERR_UNSUPPORTED;  // one row of all P shards does not fit the array

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the array's address is the current device's: the stream must belong
    // to that device
    int dev = 0, stream_dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaStreamGetDevice(st, &stream_dev) != cudaSuccess)
        return TACO_ERR_CUDA;
    if (stream_dev != dev)
        return TACO_ERR_INVALID_ARG;
    uint8_t *scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess)
        return TACO_ERR_CUDA;
    for (int64_t r0 = 0; r0 < rows; r0 += R) {
        const int64_t Rc = (rows - r0 < R) ? rows - r0 : R;
        const int64_t e = Rc * d, nb = e / block;
        const ChunkLayout L = layout(P, Rc, d, block);
        auto *x = scratch + L.x;
        auto *codes = scratch + L.codes;
        auto *alpha = reinterpret_cast<float *>(scratch + L.alpha);
        auto *scale = reinterpret_cast<float *>(scratch + L.scale);
        auto *rcodes = scratch + L.rcodes;
        auto *ralpha = reinterpret_cast<float *>(scratch + L.ralpha);
        auto *rscale = reinterpret_cast<float *>(scratch + L.rscale);
        auto *out = reinterpret_cast<float *>(scratch + L.out);

        const auto *src = static_cast<const uint8_t *>(x_host_bf16) + static_cast<size_t>(r0 * d) * 2;
        if (cudaMemcpy2DAsync(x, static_cast<size_t>(e) * 2, src, static_cast<size_t>(rows * d) * 2,
                              static_cast<size_t>(e) * 2, static_cast<size_t>(P), cudaMemcpyHostToDevice,
                              st) != cudaSuccess)
            return TACO_ERR_CUDA;
        if (taco::launch_compress(x, P * e / 128, block, e_target, eps, codes, alpha, scale, false, st) !=
            cudaSuccess)
            return TACO_ERR_CUDA;
        taco::ShardPtrs sp = {};
        for (int q = 0; q < P; ++q) {
            sp.codes[q] = codes + q * e;
            sp.alpha[q] = alpha + q * nb;
            sp.scale[q] = scale + q * nb;
        }
        if (taco::launch_taco_reduce(P, sp, nb, block, e_target, eps, rcodes, ralpha, rscale, st) != cudaSuccess ||
            taco::launch_decompress(rcodes, ralpha, rscale, e / 128, block, out, false, false, st) != cudaSuccess)
            return TACO_ERR_CUDA;
        if (cudaMemcpyAsync(out_host + r0 * d, out, static_cast<size_t>(e) * 4, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess)
            return TACO_ERR_CUDA;
    }
    return TACO_OK;
}

}  // extern "C"
