// Fused ASH + DS FP8 compressor and its inverse for sm_103a.
//
// TACO (gist.science summary of arXiv 2604.24088), 2.B.1 - 2.B.3: per block,
// energy -> adaptive pre-scale alpha -> orthogonal Hadamard rotation ->
// post-scale s keeping values inside +-448 -> E4M3 codes, fused into one
// kernel with no intermediate global-memory round trip; decompression
// inverts the rotation with both scales.
//
// Design (GB300):
//  * The tensor is viewed as nrows rows of 128 elements.  One consumer
//    thread owns one row in registers, so the 7 butterfly stages of a
//    128-point Walsh-Hadamard transform are plain register FADDs with no
//    shuffles.  A 256-element block spans two adjacent lanes and needs one
//    extra __shfl_xor stage.
//  * Every warp is an independent pipeline over 32-row tiles: lane 0 keeps
//    compress_stages<NB>() (compress) or kDStages (decompress) TMA loads
//    (cp.async.bulk.tensor, 128-byte swizzle) in flight into the warp's own
//    ring of mbarrier-guarded stages and refills a stage as soon as the warp
//    has read it.  The swizzle makes each lane's
//    row reads bank-conflict free.  No producer warp and no cross-warp
//    barrier: 8 warps per CTA leave 255 registers per thread.
//  * Each warp writes its 32 output rows into its own swizzled staging
//    buffer and stores them with TMA tensor stores.
//  * Persistent grid: one CTA per SM, warp tiles handed out round-robin.
//  * Every mbarrier wait is time-limited (device_utils.cuh); a wait that
//    runs out sets a flag readable through taco_device_error().

#include <atomic>
#include <cfloat>
#include <mutex>

#include "codec_math.cuh"
#include "device_utils.cuh"
#include "internal.h"

namespace taco {

__device__ unsigned int g_codec_error;

constexpr int kWarps = 8;              // warps per CTA, each an independent pipeline
constexpr int kThreads = kWarps * 32;
constexpr int kWarpRows = 32;          // rows per warp tile, one per lane
// TMA ring depth per warp.  Measured on GB300 in the back-to-back step
// (where the compressor also writes back the previous decompress output),
// the n=128 compressor is fastest with one stage: its next tile is loaded
// while the current one is computed (69.2 us at the headline size, against
// 76.5 with two stages and 79.0 with three).  At n=256, where a lane pair
// shares a block and each tile carries more work, two stages are 2% faster.
// The decompressor keeps three.
template <int NB> __host__ __device__ constexpr int compress_stages() { return NB == 128 ? 1 : 2; }
constexpr int kDStages = 3;
constexpr uint32_t kErrCompress = 1u;
constexpr uint32_t kErrDecompress = 2u;

// compress, per warp: stages x (two 128-byte-wide halves of 32 rows of
// bf16) + 32 rows x 128 bytes of codes
constexpr uint32_t kCHalfBytes = kWarpRows * 128;           // 4 KB
constexpr uint32_t kCStageBytes = 2 * kCHalfBytes;          // 8 KB
constexpr uint32_t kCOutBytes = kWarpRows * 128;            // 4 KB
template <int NB> __host__ __device__ constexpr uint32_t compress_warp_bytes()
{
    return compress_stages<NB>() * kCStageBytes + kCOutBytes;
}
template <int NB> __host__ __device__ constexpr uint32_t compress_smem_bytes()
{
    return 1024 + kWarps * compress_warp_bytes<NB>() + kWarps * compress_stages<NB>() * 8;
}
// decompress, per warp: kDStages x 32 rows x 128 codes + 32 rows x 512 bytes
constexpr uint32_t kDStageBytes = kWarpRows * 128;          // 4 KB
constexpr uint32_t kDOutBytes = kWarpRows * 512;            // 16 KB
constexpr uint32_t kDWarpBytes = kDStages * kDStageBytes + kDOutBytes;  // 28 KB
static_assert(compress_warp_bytes<128>() % 1024 == 0 && compress_warp_bytes<256>() % 1024 == 0 &&
                  kDWarpBytes % 1024 == 0,
              "swizzle atoms need 1 KB alignment");
constexpr uint32_t kDSmemBytes = 1024 + kWarps * kDWarpBytes + kWarps * kDStages * 8;

// ===================================================================== //
//                              compressor                               //
// ===================================================================== //

// Each warp streams its own 32-row tiles: warp tile t covers rows
// 32t .. 32t + 31; the warps of the grid take tiles round-robin.  Lane 0
// keeps compress_stages<NB>() TMA loads in flight and refills a stage as soon as the warp
// has read it.

// One 32-row bf16 input tile (two 64-column boxes) into a pipeline stage.
// The input is read once: evict-first keeps L2 for the codes this kernel
// writes, which the shard reduce reads next.
__device__ __forceinline__ void load_input_tile(uint32_t dst, const CUtensorMap *x_map, int32_t y, uint32_t full)
{
    const uint64_t pol = policy_evict_first();
    tma_load_2d_hint(dst, x_map, 0, y, full, pol);
    tma_load_2d_hint(dst + kCHalfBytes, x_map, 64, y, full, pol);
}

// FMT_INT8: INT8 codes with Q_max = 127 (the fallback format); otherwise
// E4M3 codes with Q_max = 448.
template <int NB, bool FMT_INT8>
__global__ void __launch_bounds__(kThreads, 1)
    taco_compress_kernel(const __grid_constant__ CUtensorMap x_map,
                         const __grid_constant__ CUtensorMap c_map, float *__restrict__ alpha_out,
                         float *__restrict__ scale_out, int64_t nrows, float e_target, float eps)
{
    constexpr int G = NB / 128;  // lanes per block
    constexpr int kCStages = compress_stages<NB>();
    constexpr uint32_t kCWarpBytes = compress_warp_bytes<NB>();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t wbase = base + warp * kCWarpBytes;
    const uint32_t outw = wbase + kCStages * kCStageBytes;
    const uint32_t bars = base + kWarps * kCWarpBytes + warp * kCStages * 8;
    // 32-bit row and tile indices (the host rejects nrows >= 2^31): fewer
    // registers in a kernel that uses all 255
    const int nrows32 = static_cast<int>(nrows);
    const int ntiles = (nrows32 + kWarpRows - 1) / kWarpRows;
    const int gw = blockIdx.x * kWarps + warp;
    const int W = gridDim.x * kWarps;

    pdl_wait();
    int issued = 0;
    if (lane == 0) {
        tma_prefetch_map(&x_map);
        for (int s = 0; s < kCStages; ++s)
            mbar_init(bars + 8 * s, 1);
        fence_barrier_init();
        for (; issued < kCStages && gw + issued * W < ntiles; ++issued) {
            const int32_t y = static_cast<int32_t>((gw + issued * W) * kWarpRows);
            const uint32_t dst = wbase + issued * kCStageBytes, full = bars + 8 * issued;
            mbar_arrive_expect_tx(full, kCStageBytes);
            load_input_tile(dst, &x_map, y, full);
        }
    }
    __syncwarp();

    const uint32_t swz = static_cast<uint32_t>(lane & 7) << 4;
    const uint32_t orow = outw + lane * 128;
    const float c = BlockConst<NB>::c;
    int it = 0;
    for (int t = gw; t < ntiles; t += W, ++it) {
        const int s = it % kCStages;
        // warp-uniform: if any lane's wait runs out, the whole warp stops
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bars + 8 * s, (it / kCStages) & 1))) {
            if (lane == 0)
                atomicOr(&g_codec_error, kErrCompress);
            break;
        }
        // Lane l reads row l of the stage: half h holds elements 64h .. 64h+63,
        // and 16-byte chunk j of a 128-byte row sits at chunk j ^ (l & 7).
        const uint32_t rowp = wbase + s * kCStageBytes + lane * 128;
        float2 v[64];
        float2 acc[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 q = lds128(rowp + h * kCHalfBytes + ((static_cast<uint32_t>(j) << 4) ^ swz));
                // step 1 (energy, exact squares of bf16 values) and the
                // bit-0 butterfly stage of step 3
                unpack8_stage1(q, v, h * 32 + j * 4, acc, h == 0 && j < 2);
            }
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i)
                acc[i] = __fadd2_rn(acc[i], acc[i + w]);
        float ss = acc[0].x + acc[0].y;
        // every loaded value has been consumed: refill the stage
        __syncwarp();
        if (lane == 0) {
            const int nt = gw + (it + kCStages) * W;
            if (nt < ntiles) {
                fence_proxy_async_smem();
                const uint32_t dst = wbase + s * kCStageBytes, full = bars + 8 * s;
                const int32_t y = static_cast<int32_t>(nt * kWarpRows);
                mbar_arrive_expect_tx(full, kCStageBytes);
                load_input_tile(dst, &x_map, y, full);
                ++issued;
            }
        }

        // step 3: remaining butterfly stages (alpha and 1/sqrt(n) are applied
        // below; at n = 128 the last stage is fused with that scaling)
        float mh;
        if constexpr (G == 2) {
            fwht128_upper(v);
            fwht_pair_stage(v, lane);
            ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
            mh = max_abs128(v);
            mh = fmaxf(mh, __shfl_xor_sync(0xFFFFFFFFu, mh, 1));
        } else {
            fwht128_upper_but_last(v);
            mh = max_abs_last_stage(v);
        }

        // step 2: alpha = sqrt(E / (m + eps));  step 4: s = 448 / max|y|
        const float m = ss * BlockConst<NB>::inv_n;
        const float alpha = sqrtf(e_target / (m + eps));
        const float ac = alpha * c;
        const float M = ac * mh;
        constexpr float kQmax = FMT_INT8 ? 127.0f : 448.0f;
        const float scale = (M > 0.0f) ? fminf(kQmax / M, FLT_MAX) : 1.0f;
        float k = ac * scale;
        if (!(k <= FLT_MAX)) {  // block of tiny values: apply the two factors separately
            const float2 ac2 = make_float2(ac, ac);
#pragma unroll
            for (int i = 0; i < 64; ++i)
                v[i] = __fmul2_rn(v[i], ac2);
            k = scale;
        }
        const float2 k2 = make_float2(k, k);
        if constexpr (G == 1)
            last_stage_scaled(v, k2);  // v now holds y * s

        // step 5: codes = E4M3(y * s) into the warp's swizzled staging rows
        if (lane == 0)
            bulk_wait_read_all();  // the previous store from this buffer is done reading
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t w0, w1, w2, w3;
            if constexpr (FMT_INT8 && G == 1) {
                encode8_s8_prescaled(&v[8 * j], w0, w1);
                encode8_s8_prescaled(&v[8 * j + 4], w2, w3);
            } else if constexpr (FMT_INT8) {
                encode8_s8(&v[8 * j], k2, w0, w1);
                encode8_s8(&v[8 * j + 4], k2, w2, w3);
            } else if constexpr (G == 1) {
                encode8_prescaled(&v[8 * j], w0, w1);
                encode8_prescaled(&v[8 * j + 4], w2, w3);
            } else {
                encode8(&v[8 * j], k2, w0, w1);
                encode8(&v[8 * j + 4], k2, w2, w3);
            }
            sts128(orow + ((static_cast<uint32_t>(j) << 4) ^ swz), w0, w1, w2, w3);
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int wrow = t * kWarpRows;
        if (lane == 0) {
            tma_store_2d(&c_map, 0, static_cast<int32_t>(wrow), outw);
            bulk_commit();
        }
        const int grow = wrow + lane;
        if (grow < nrows32 && (lane % G) == 0) {
            alpha_out[grow / G] = alpha;
            scale_out[grow / G] = scale;
        }
    }
    if (lane == 0) {
        // leave no copy in flight into or out of this CTA's shared memory
        for (int k = it; k < issued; ++k)
            mbar_wait(bars + 8 * (k % kCStages), (k / kCStages) & 1);
        bulk_wait_all();
    }
}

// ===================================================================== //
//                             decompressor                              //
// ===================================================================== //

template <int NB, bool BF16OUT, bool FMT_INT8>
__global__ void __launch_bounds__(kThreads, 1)
    taco_decompress_kernel(const __grid_constant__ CUtensorMap c_map,
                           const __grid_constant__ CUtensorMap o_map, const float *__restrict__ alpha,
                           const float *__restrict__ scale, int64_t nrows)
{
    constexpr int G = NB / 128;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t wbase = base + warp * kDWarpBytes;
    const uint32_t outw = wbase + kDStages * kDStageBytes;
    const uint32_t bars = base + kWarps * kDWarpBytes + warp * kDStages * 8;
    const int64_t ntiles = (nrows + kWarpRows - 1) / kWarpRows;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    const int64_t W = static_cast<int64_t>(gridDim.x) * kWarps;

    pdl_wait();
    int issued = 0;
    if (lane == 0) {
        tma_prefetch_map(&c_map);
        for (int s = 0; s < kDStages; ++s)
            mbar_init(bars + 8 * s, 1);
        fence_barrier_init();
        // the codes are read once (evict-first L2 policy)
        for (; issued < kDStages && gw + issued * W < ntiles; ++issued) {
            const uint32_t full = bars + 8 * issued;
            mbar_arrive_expect_tx(full, kDStageBytes);
            tma_load_2d_hint(wbase + issued * kDStageBytes, &c_map, 0,
                             static_cast<int32_t>((gw + issued * W) * kWarpRows), full, policy_evict_first());
        }
    }
    __syncwarp();

    const uint32_t swz = static_cast<uint32_t>(lane & 7) << 4;
    // the block scalars of a tile are loaded one tile ahead
    auto tile_block = [&](int64_t t) {
        const int64_t grow = t * kWarpRows + lane;
        return (grow < nrows ? grow : nrows - 1) / G;
    };
    float a_next = 1.0f, sc_next = 1.0f;
    if (gw < ntiles) {
        a_next = __ldg(alpha + tile_block(gw));
        sc_next = __ldg(scale + tile_block(gw));
    }
    int it = 0;
    for (int64_t t = gw; t < ntiles; t += W, ++it) {
        const int s = it % kDStages;
        const int64_t wrow = t * kWarpRows;
        const float a = a_next, sc = sc_next;
        if (t + W < ntiles) {
            a_next = __ldg(alpha + tile_block(t + W));
            sc_next = __ldg(scale + tile_block(t + W));
        }
        // warp-uniform: if any lane's wait runs out, the whole warp stops
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bars + 8 * s, (it / kDStages) & 1))) {
            if (lane == 0)
                atomicOr(&g_codec_error, kErrDecompress);
            break;
        }
        const uint32_t rowp = wbase + s * kDStageBytes + lane * 128;
        float2 v[64];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 q = lds128(rowp + ((static_cast<uint32_t>(j) << 4) ^ swz));
            if constexpr (FMT_INT8)
                decode16_stage1_s8(q, v, j);
            else
                decode16_stage1(q, v, j);
        }
        if constexpr (G == 2)
            fwht128_upper(v);  // consumes every decoded value
        else
            fwht128_upper_but_last(v);  // the last stage is fused with the scaling below
        __syncwarp();
        if (lane == 0) {
            const int64_t nt = gw + static_cast<int64_t>(it + kDStages) * W;
            if (nt < ntiles) {
                fence_proxy_async_smem();
                const uint32_t full = bars + 8 * s;
                mbar_arrive_expect_tx(full, kDStageBytes);
                tma_load_2d_hint(wbase + s * kDStageBytes, &c_map, 0, static_cast<int32_t>(nt * kWarpRows), full,
                                 policy_evict_first());
                ++issued;
            }
        }
        if constexpr (G == 2)
            fwht_pair_stage(v, lane);

        // out = c H(decode) / (s alpha)
        const float2 k2 = decompress_multiplier<NB>(v, sc, a);
        if constexpr (G == 1)
            last_stage_scaled(v, k2);
        if (lane == 0)
            bulk_wait_read_all();
        __syncwarp();
        stage_output_row<BF16OUT, G == 1>(v, k2, outw, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            constexpr int nbox = BF16OUT ? 2 : 4;
            constexpr int box_inner = BF16OUT ? 64 : 32;
            // written once and not read again by this path: evict-first
            // lets L2 write the tile back now instead of leaving it dirty
            // for the next kernel to flush
            const uint64_t pol = policy_evict_first();
#pragma unroll
            for (int b = 0; b < nbox; ++b)
                tma_store_2d_hint(&o_map, b * box_inner, static_cast<int32_t>(wrow), outw + b * 4096, pol);
            bulk_commit();
        }
    }
    if (lane == 0) {
        for (int k = it; k < issued; ++k)
            mbar_wait(bars + 8 * (k % kDStages), (k / kDStages) & 1);
        bulk_wait_all();
    }
}

// ===================================================================== //
//                          watchdog self-test                           //
// ===================================================================== //

constexpr uint32_t kErrSelftest = 16u;

// One warp waits, with the codec kernels' time-limited wait, on an mbarrier
// that nothing ever arrives on.  The wait must give up (after about a
// second) and the kernel must record that in the watchdog flags and return,
// leaving the context usable: the path a stalled TMA copy would take.
__global__ void __launch_bounds__(32) watchdog_selftest_kernel()
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncwarp();
    const bool done = __all_sync(0xFFFFFFFFu, mbar_wait(b, 0));
    if (!done && threadIdx.x == 0)
        atomicOr(&g_codec_error, kErrSelftest);
}

// ===================================================================== //
//                                 host                                  //
// ===================================================================== //

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

constexpr int kMaxDevices = 64;

// Raises a kernel's dynamic shared-memory limit once per device.  The flag
// is atomic because host threads may make their first launch concurrently;
// setting the attribute twice is harmless.
template <typename K>
cudaError_t ensure_smem(K kernel, uint32_t bytes, int device, std::atomic<bool> *done)
{
    if (done[device].load(std::memory_order_acquire))
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (e == cudaSuccess)
        done[device].store(true, std::memory_order_release);
    return e;
}

}  // namespace

int encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base, uint64_t inner,
                         uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                         uint32_t box_rows, CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return -1;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -2;
}

namespace {

template <int NB, bool I8>
cudaError_t run_compress(const CUtensorMap &xm, const CUtensorMap &cm, float *alpha, float *scale,
                         int64_t nrows, float e_target, float eps, int grid, cudaStream_t stream, int device)
{
    static std::atomic<bool> set[kMaxDevices];
    constexpr uint32_t smem = compress_smem_bytes<NB>();
    cudaError_t e = ensure_smem(taco_compress_kernel<NB, I8>, smem, device, set);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(taco_compress_kernel<NB, I8>, grid, kThreads, smem, stream, xm, cm, alpha, scale, nrows,
                      e_target, eps);
}

template <int NB, bool BF, bool I8>
cudaError_t run_decompress(const CUtensorMap &cm, const CUtensorMap &om, const float *alpha,
                           const float *scale, int64_t nrows, int grid, cudaStream_t stream, int device)
{
    static std::atomic<bool> set[kMaxDevices];
    cudaError_t e = ensure_smem(taco_decompress_kernel<NB, BF, I8>, kDSmemBytes, device, set);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(taco_decompress_kernel<NB, BF, I8>, grid, kThreads, kDSmemBytes, stream, cm, om, alpha,
                      scale, nrows);
}

}  // namespace

cudaError_t launch_compress(const void *x_bf16, int64_t nrows, int block, float e_target, float eps,
                            uint8_t *codes, float *alpha, float *scale, bool int8_codes, cudaStream_t stream)
{
    if (nrows > (int64_t(1) << 31) - 256)  // the kernel's row and tile indices are 32-bit
        return cudaErrorInvalidValue;
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess)
        return e;
    CUtensorMap xm, cm;
    if (encode_tensor_map_2d(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(x_bf16), 128,
                             nrows, 256, 64, kWarpRows) != 0 ||
        encode_tensor_map_2d(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, 128, nrows, 128, 128, 32) != 0)
        return cudaErrorInvalidValue;
    const int64_t ctas = (nrows + kWarps * kWarpRows - 1) / (kWarps * kWarpRows);
    const int grid = static_cast<int>(ctas < di.num_sms ? ctas : di.num_sms);
    if (block == 128)
        return int8_codes ? run_compress<128, true>(xm, cm, alpha, scale, nrows, e_target, eps, grid, stream, di.device)
                          : run_compress<128, false>(xm, cm, alpha, scale, nrows, e_target, eps, grid, stream,
                                                     di.device);
    return int8_codes ? run_compress<256, true>(xm, cm, alpha, scale, nrows, e_target, eps, grid, stream, di.device)
                      : run_compress<256, false>(xm, cm, alpha, scale, nrows, e_target, eps, grid, stream, di.device);
}

cudaError_t launch_decompress(const uint8_t *codes, const float *alpha, const float *scale, int64_t nrows,
                              int block, void *out, bool out_bf16, bool int8_codes, cudaStream_t stream)
{
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess)
        return e;
    CUtensorMap cm, om;
    int rc = encode_tensor_map_2d(&cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<uint8_t *>(codes), 128,
                                  nrows, 128, 128, kWarpRows);
    if (out_bf16)
        rc |= encode_tensor_map_2d(&om, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, 128, nrows, 256, 64, 32);
    else
        rc |= encode_tensor_map_2d(&om, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out, 128, nrows, 512, 32, 32);
    if (rc != 0)
        return cudaErrorInvalidValue;
    const int64_t ctas = (nrows + kWarps * kWarpRows - 1) / (kWarps * kWarpRows);
    const int grid = static_cast<int>(ctas < di.num_sms ? ctas : di.num_sms);
    const int dev = di.device;
    if (block == 128) {
        if (int8_codes)
            return out_bf16 ? run_decompress<128, true, true>(cm, om, alpha, scale, nrows, grid, stream, dev)
                            : run_decompress<128, false, true>(cm, om, alpha, scale, nrows, grid, stream, dev);
        return out_bf16 ? run_decompress<128, true, false>(cm, om, alpha, scale, nrows, grid, stream, dev)
                        : run_decompress<128, false, false>(cm, om, alpha, scale, nrows, grid, stream, dev);
    }
    if (int8_codes)
        return out_bf16 ? run_decompress<256, true, true>(cm, om, alpha, scale, nrows, grid, stream, dev)
                        : run_decompress<256, false, true>(cm, om, alpha, scale, nrows, grid, stream, dev);
    return out_bf16 ? run_decompress<256, true, false>(cm, om, alpha, scale, nrows, grid, stream, dev)
                    : run_decompress<256, false, false>(cm, om, alpha, scale, nrows, grid, stream, dev);
}

cudaError_t launch_watchdog_selftest(cudaStream_t stream)
{
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

cudaError_t read_codec_error(uint32_t *flags, bool clear)
{
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_codec_error, sizeof v);
    if (e != cudaSuccess)
        return e;
    *flags = v;
    if (clear) {
        v = 0;
        e = cudaMemcpyToSymbol(g_codec_error, &v, sizeof v);
    }
    return e;
}

}  // namespace taco
