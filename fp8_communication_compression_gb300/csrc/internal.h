// Host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace taco {

// Per-device facts the launchers need (cached on first use).
struct DeviceInfo {
    int device;
    int num_sms;
    int max_smem_optin;
};
cudaError_t current_device_info(DeviceInfo *out);

// cuTensorMapEncodeTiled, resolved through the runtime's driver entry point
// (128-byte swizzle unless asked otherwise).  Returns 0 on success.
int encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, void *base, uint64_t inner,
                         uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner,
                         uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// Kernels working on the "128-view" of a TACO tensor: nrows rows of 128
// elements; a block of n elements spans n / 128 consecutive rows.
// int8_codes selects the INT8 code format (Q_max 127) instead of E4M3.
cudaError_t launch_compress(const void *x_bf16, int64_t nrows, int block, float e_target, float eps,
                            uint8_t *codes, float *alpha, float *scale, bool int8_codes,
                            cudaStream_t stream);
cudaError_t launch_decompress(const uint8_t *codes, const float *alpha, const float *scale,
                              int64_t nrows, int block, void *out, bool out_bf16, bool int8_codes,
                              cudaStream_t stream);

// Direct-load kernels (no Hadamard on their path).
struct ShardPtrs {
    const uint8_t *codes[16];
    const float *alpha[16];
    const float *scale[16];
};
cudaError_t launch_taco_reduce(int P, const ShardPtrs &in, int64_t nblocks, int block, float e_target,
                               float eps, uint8_t *out_codes, float *out_alpha, float *out_scale,
                               cudaStream_t stream);
cudaError_t launch_reduce_decompress(int P, const ShardPtrs &in, int64_t nrows, int block, float e_target,
                                     float eps, uint8_t *out_codes, float *out_alpha, float *out_scale,
                                     void *out, bool out_bf16, cudaStream_t stream);
cudaError_t launch_agoq_accumulate(uint8_t *codes, float *scale, const void *grad_bf16, int64_t n,
                                   int block, cudaStream_t stream);
cudaError_t launch_agoq_reduce(int P, const ShardPtrs &in, int64_t n, int block, uint8_t *out_codes,
                               float *out_scale, cudaStream_t stream);

cudaError_t launch_laaq_quantize(const void *x_bf16, int64_t n, int block, int bits, uint8_t *packed,
                                 float *scale, cudaStream_t stream);
cudaError_t launch_laaq_dequantize(const uint8_t *packed, const float *scale, int64_t n, int block, int bits,
                                   void *out, bool out_bf16, bool silu, cudaStream_t stream);
// RMSNorm of each row of d values (d % block == 0) recomputed from the
// stored quantised input: y = x_hat / sqrt(mean(x_hat^2) + eps) * gamma.
cudaError_t launch_laaq_rmsnorm(const uint8_t *packed, const float *scale, int64_t rows, int64_t d, int block,
                                int bits, const float *gamma, float eps, void *out, bool out_bf16,
                                cudaStream_t stream);

cudaError_t launch_e4m3_encode(const float *x, int64_t n, uint8_t *codes, cudaStream_t stream);

// Chunked host-buffer pipeline of the two-shot local path (host_pipeline.cu).
struct HostPipeline;
int host_pipeline_max_chunks();
cudaError_t host_pipeline_create(int P, int64_t rows, int64_t d, int block, int chunks, bool out_bf16,
                                 HostPipeline **out, uint64_t *workspace_bytes);
void host_pipeline_destroy(HostPipeline *p);
int host_pipeline_device(const HostPipeline *p);
uint64_t host_pipeline_workspace(const HostPipeline *p);
cudaError_t host_pipeline_run(HostPipeline *p, const void *x_host, void *out_host, void *workspace, float e_target,
                              float eps, cudaStream_t stream);

// Tensor-core GEMM Y = A B^T (bf16, fp32 accumulate) with the ASH + DS
// compressor in its epilogue (gemm_compress.cu): M % 128 == 0,
// N % 128 == 0, K % 64 == 0, block 128.  y_out (fp32 [M][N]) may be null.
// workspace (workspace_bytes, 256-byte aligned, zeroed before its first
// use) holds the split tail's partial sums; null or too small: no split.
cudaError_t launch_gemm_compress(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                 float e_target, float eps, uint8_t *codes, float *alpha, float *scale,
                                 float *y_out, void *workspace, uint64_t workspace_bytes, cudaStream_t stream);
// The same GEMM with the AGoQ accumulation into an FP8 main gradient
// ([M][N] codes and [M][N / 128] multipliers, in place) in its epilogue.
cudaError_t launch_gemm_agoq_accumulate(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                        uint8_t *main_codes, float *main_scale, float *y_out, void *workspace,
                                        uint64_t workspace_bytes, cudaStream_t stream);
// The same GEMM with AGoQ's LAAQ activation quantisation of its output in
// its epilogue: blocks of 128 along each row, `bits` (4, 5, 6 or 8) bits a
// code, packed [M][N * bits / 8] and multipliers [M][N / 128].
cudaError_t launch_gemm_laaq_quantize(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                      int bits, uint8_t *packed, float *scale, float *y_out, void *workspace,
                                      uint64_t workspace_bytes, cudaStream_t stream);
// Workspace the split tail of an M x N x K GEMM takes on the current device
// (0 when it takes none).
cudaError_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, uint64_t *bytes);

cudaError_t launch_watchdog_selftest(cudaStream_t stream);
cudaError_t read_codec_error(uint32_t *flags, bool clear);
cudaError_t read_gemm_error(uint32_t *flags, bool clear);

// Launches `kernel` with programmatic stream serialization allowed, so that
// it can be scheduled while the previous kernel in the stream drains (every
// kernel of this library waits for its predecessor with griddepcontrol.wait
// before reading inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

} // namespace taco
