// The E4M3 encoder of the compressor on its own: fp32 values -> E4M3FN
// codes with round-to-nearest-even and saturation at +-448 (TACO, gist.science
// summary of arXiv 2604.24088, 2.A: the FP8 format the codes use).  It runs
// the same device conversion the codec kernels use, so a caller can encode
// values it has scaled itself, and the conversion can be checked value by
// value against the format's definition.

#include "device_utils.cuh"
#include "internal.h"

namespace taco {

namespace {

constexpr int kEThreads = 256;

// Each thread encodes groups of 8 values: two 16-byte loads, one 8-byte
// store.  The last n % 8 values are encoded one by one.
__global__ void __launch_bounds__(kEThreads)
    e4m3_encode_kernel(const float *__restrict__ x, int64_t n, uint8_t *__restrict__ codes)
{
    pdl_wait();
    const int64_t groups = n / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups; g += stride) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(x) + 2 * g);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(x) + 2 * g + 1);
        reinterpret_cast<uint2 *>(codes)[g] =
            make_uint2(f32x4_to_e4m3x4(a.x, a.y, a.z, a.w), f32x4_to_e4m3x4(b.x, b.y, b.z, b.w));
    }
    if (blockIdx.x == 0 && threadIdx.x < n - 8 * groups) {
        const int64_t i = 8 * groups + threadIdx.x;
        codes[i] = static_cast<uint8_t>(f32x2_to_e4m3x2(x[i], 0.0f) & 0xFFu);
    }
}

}  // namespace

cudaError_t launch_e4m3_encode(const float *x, int64_t n, uint8_t *codes, cudaStream_t stream)
{
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, e4m3_encode_kernel, kEThreads, 0)) !=
        cudaSuccess)
        return e;
    const int64_t need = (n / 8 + kEThreads - 1) / kEThreads;
    const int64_t cap = static_cast<int64_t>(di.num_sms) * (per_sm < 1 ? 1 : per_sm);
    const int grid = static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
    return launch_pdl(e4m3_encode_kernel, grid, kEThreads, 0, stream, x, n, codes);
}

}  // namespace taco
