/*
 * taco.h - C ABI of the GB300 (sm_103a) FP8 communication-compression library.
 *
 * The operations follow two web summaries of papers:
 *   [TACO] "TACO: Efficient Communication Compression of Intermediate Tensors
 *          for Scalable Tensor-Parallel LLM Training" (gist.science summary
 *          of arXiv 2604.24088)
 *   [AGoQ] "AGoQ: Activation and Gradient Quantization for Memory-Efficient
 *          Distributed Training of LLMs" (gist.science summary of arXiv
 *          2605.00539)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Memory: every pointer argument is a DEVICE pointer unless stated
 *    otherwise.  The caller allocates and owns every buffer; the library
 *    never allocates, frees or synchronises, and keeps no state beyond a
 *    per-device cache of attributes and kernel settings.  (The host
 *    pipeline's create and destroy calls create and release CUDA streams
 *    and events, and nothing else.)
 *  - Execution: each call validates its arguments on the host, then enqueues
 *    its work on `stream` and returns; results are ready when the stream
 *    reaches that point.  Device-buffer calls enqueue one kernel, except
 *    taco_reduce_decompress (two); the host-buffer calls enqueue copies and
 *    kernels per row chunk.  A NULL stream is the legacy
 *    default stream.
 *  - Layout: tensors are row-major and contiguous.  A "block" is a run of
 *    `block` consecutive elements of a row; `d % block == 0`, so a tensor
 *    of rows x d elements holds nb = rows * d / block blocks, stored one after
 *    another.  Per-block scalars (alpha, scale) are fp32 arrays of nb values
 *    in the same order.  FP8 codes are E4M3FN bit patterns, one byte each
 *    (viewable as torch.float8_e4m3fn); bf16 data is passed as raw 16-bit
 *    patterns.
 *  - Alignment: bf16, code and fp32 output buffers must be 16-byte aligned;
 *    alpha and scale arrays 4-byte aligned.
 *  - Aliasing: outputs must not overlap inputs, except where an argument is
 *    documented as in/out.
 *  - Errors: a bad argument returns a status and launches nothing.  A
 *    failed launch returns TACO_ERR_CUDA.  Nothing aborts and no C++
 *    exception crosses the ABI.  Kernels never wait without a time limit;
 *    a wait that runs out records a flag read by taco_device_error().
 *  - Empty input (rows == 0 or n == 0) returns TACO_OK without a launch.
 *  - Size limit: a TACO call takes at most 2^31 - 256 rows of 128 elements
 *    (rows * d / 128), more than any GPU memory holds; larger calls return
 *    TACO_ERR_UNSUPPORTED.
 *  - Inputs must be finite; NaN or Inf input gives unspecified codes
 *    (taco_e4m3_encode states its own handling of them).
 */
#ifndef TACO_H
#define TACO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that the header needs no
 * CUDA include. */
typedef struct CUstream_st *taco_stream_t;

typedef enum {
    TACO_OK = 0,
    TACO_ERR_INVALID_ARG = 1, /* null pointer, bad size, overlap, non-positive e_target/eps */
    TACO_ERR_UNSUPPORTED = 2, /* block size or shard count outside the supported set */
    TACO_ERR_MISALIGNED = 3,  /* pointer alignment below the stated minimum */
    TACO_ERR_CUDA = 4,        /* the CUDA runtime reported an error */
} taco_status;

#define TACO_ABI_VERSION 1
#define TACO_QMAX 448.0f
#define TACO_MAX_SHARDS 16

/* Human-readable name of a status; never NULL. */
const char *taco_status_string(taco_status status);

/* Returns TACO_ABI_VERSION of the loaded library. */
int taco_abi_version(void);

/* Block sizes the TACO calls accept: 128 and 256. */
int taco_block_supported(int32_t block);

/*
 * taco_compress - fused ASH + DS FP8 compressor.
 * [TACO] 2.B.1 (ASH), 2.B.2 (DS), 2.B.3 (fused operator).  For every block:
 *   m      = mean(x^2)                          (block energy)
 *   alpha  = sqrt(e_target / (m + eps))         (pre-transform scale)
 *   y      = (1/sqrt(block)) H (alpha x)        (Sylvester-order Hadamard)
 *   scale  = 448 / max|y|   (1 if y == 0)       (post-transform scale)
 *   codes  = E4M3(y * scale), round to nearest even, saturating at +-448
 * in one pass, with no intermediate global-memory round trip.
 *
 *  x_bf16   in   bf16 [rows, d]
 *  rows, d       rows >= 0, d > 0, d % block == 0
 *  block         128 or 256
 *  e_target      target block energy, > 0 (finite)
 *  eps           energy floor, > 0 (finite)
 *  codes    out  uint8 [rows, d] E4M3FN codes
 *  alpha    out  fp32 [nb]
 *  scale    out  fp32 [nb]
 */
taco_status taco_compress(const void *x_bf16, int64_t rows, int64_t d, int32_t block,
                          float e_target, float eps, uint8_t *codes, float *alpha,
                          float *scale, taco_stream_t stream);

/*
 * taco_decompress - exact inverse of the compressor up to the FP8 rounding.
 * [TACO] 2.B.2 reconstruction with both scales:
 *   out = (1/sqrt(block)) H (decode(codes) / scale) / alpha
 *
 *  codes, alpha, scale   in   as produced by taco_compress
 *  out                   out  [rows, d]: fp32, or bf16 (round to nearest
 *                             even) when out_is_bf16 != 0
 */
taco_status taco_decompress(const uint8_t *codes, const float *alpha, const float *scale,
                            int64_t rows, int64_t d, int32_t block, void *out,
                            int32_t out_is_bf16, taco_stream_t stream);

/*
 * taco_compress_int8 / taco_decompress_int8 - the same ASH + DS codec with
 * INT8 codes, the fallback [TACO] 5 names for hardware without native FP8:
 *   scale  = 127 / max|y|   (1 if y == 0)
 *   codes  = round-to-nearest-even(y * scale), in [-127, 127]
 *   out    = (1/sqrt(block)) H (codes / scale) / alpha
 * Arguments, layouts and errors as taco_compress / taco_decompress; codes
 * are int8 [rows, d].
 */
taco_status taco_compress_int8(const void *x_bf16, int64_t rows, int64_t d, int32_t block,
                               float e_target, float eps, int8_t *codes, float *alpha,
                               float *scale, taco_stream_t stream);
taco_status taco_decompress_int8(const int8_t *codes, const float *alpha, const float *scale,
                                 int64_t rows, int64_t d, int32_t block, void *out,
                                 int32_t out_is_bf16, taco_stream_t stream);

/*
 * taco_reduce_shards - local step of the two-shot AllReduce
 * ([TACO] 2.B.3 ReduceScatter + AllGather; [AGoQ] 2.B "local reduce in
 * FP32"): P compressed shards of the same [rows, d] region, all resident in
 * this GPU's memory, are dequantised, summed in FP32 and requantised with
 * the compressor above.  Result = compress(sum_p decompress(shard p)); it is
 * computed in the Hadamard domain, where the sum of the P reconstructions and
 * the compressor's forward rotation cancel (c H c H = I), so no rotation is
 * applied.
 *
 *  P                      1 .. TACO_MAX_SHARDS
 *  codes, alpha, scale    in   HOST arrays of P device pointers, shard p
 *                              laid out as taco_compress's outputs
 *  out_codes, out_alpha,  out  the compressed sum, same layout
 *  out_scale
 */
taco_status taco_reduce_shards(int32_t P, const uint8_t *const *codes,
                               const float *const *alpha, const float *const *scale,
                               int64_t rows, int64_t d, int32_t block, float e_target,
                               float eps, uint8_t *out_codes, float *out_alpha,
                               float *out_scale, taco_stream_t stream);

/*
 * taco_reduce_decompress - taco_reduce_shards and taco_decompress of its
 * result in one call.  The rank that reduces in the two-shot AllReduce
 * ([TACO] 2.B.3) both sends the compressed sum (AllGather payload) and
 * needs its reconstruction.  The call runs the shard-reduce kernel and the
 * decompress kernel back to back on `stream` (one-pass kernels measured
 * slower on this GPU), so out_codes / out_alpha / out_scale equal
 * taco_reduce_shards's outputs and `out` equals taco_decompress of them,
 * bit for bit.
 *
 *  P, codes, alpha, scale,          as taco_reduce_shards
 *  rows, d, block, e_target, eps
 *  out_codes, out_alpha, out_scale  out  the compressed sum
 *  out                              out  [rows, d] fp32, or bf16 when
 *                                        out_is_bf16 != 0
 */
taco_status taco_reduce_decompress(int32_t P, const uint8_t *const *codes,
                                   const float *const *alpha, const float *const *scale,
                                   int64_t rows, int64_t d, int32_t block, float e_target,
                                   float eps, uint8_t *out_codes, float *out_alpha,
                                   float *out_scale, void *out, int32_t out_is_bf16,
                                   taco_stream_t stream);

/*
 * agoq_fp8_accumulate - QuanGrad local accumulation, in place.
 * [AGoQ] 2.B: per block of `block` elements, in FP32 arithmetic,
 *   g       = decode(main_codes) * main_scale + grad   (rounded multiply,
 *                                                       then rounded add)
 *   codes'  = E4M3(g * (448 / max|g|))
 *   scale'  = max|g| / 448                             (1 if g == 0)
 * The stored AGoQ scale is the dequantisation multiplier: an element's
 * value is decode(code) * scale.  A zero gradient is codes 0 with scale 1.
 *
 *  main_codes  in/out  uint8 [n]
 *  main_scale  in/out  fp32 [n / block] dequantisation multipliers
 *  grad_bf16   in      bf16 [n] micro-batch gradient
 *  n                   n >= 0, n % block == 0
 *  block               128 or 256
 */
taco_status agoq_fp8_accumulate(uint8_t *main_codes, float *main_scale, const void *grad_bf16,
                                int64_t n, int32_t block, taco_stream_t stream);

/*
 * agoq_reduce_shards - precision-preserving all-reduce, local step.
 * [AGoQ] 2.B step 2: S = sum_p decode(codes_p) * scale_p, each term a
 * rounded FP32 multiply, summed in FP32 in shard order, then requantised
 * per block as in agoq_fp8_accumulate (a sum, not a mean).
 *
 *  codes, scale      in   HOST arrays of P device pointers (uint8 [n],
 *                         fp32 [n / block])
 *  out_codes         out  uint8 [n]
 *  out_scale         out  fp32 [n / block]
 */
taco_status agoq_reduce_shards(int32_t P, const uint8_t *const *codes, const float *const *scale,
                               int64_t n, int32_t block, uint8_t *out_codes, float *out_scale,
                               taco_stream_t stream);

/*
 * agoq_laaq_quantize / agoq_laaq_dequantize - block-wise activation codec of
 * AGoQ's layer-aware activation quantisation ([AGoQ] 2.A: 4-bit codes, with
 * 5, 6 or 8 bits where the pipeline-stage compensation allows).  Per block,
 * in fp32 with every operation rounded:
 *   amax = max|x|,  qmax = 2^(bits-1) - 1,  q = qmax / amax,
 *   code = clamp(round-to-nearest-even(x * q), -qmax, qmax),
 *   scale = amax / qmax (1 for an all-zero block),  x_hat = code * scale.
 * Codes are two's complement, packed little-endian: element i occupies bits
 * i*bits .. i*bits + bits - 1 of `packed` (bit j is bit j % 8 of byte j / 8).
 *
 *  x_bf16   in   bf16 [n], 16-byte aligned
 *  n             n >= 0, n % block == 0
 *  block         32, 64, 128 or 256
 *  bits          4, 5, 6 or 8
 *  packed   out  uint8 [n * bits / 8], 16-byte aligned
 *  scale    out  fp32 [n / block]
 *  out      out  [n] fp32, or bf16 (round to nearest even) when out_is_bf16
 */
taco_status agoq_laaq_quantize(const void *x_bf16, int64_t n, int32_t block, int32_t bits,
                               uint8_t *packed, float *scale, taco_stream_t stream);
taco_status agoq_laaq_dequantize(const uint8_t *packed, const float *scale, int64_t n,
                                 int32_t block, int32_t bits, void *out, int32_t out_is_bf16,
                                 taco_stream_t stream);

/*
 * agoq_laaq_dequantize_silu / agoq_laaq_dequantize_rmsnorm - an operator's
 * output recomputed from its stored quantised input ([AGoQ] 2.A: for
 * RMSNorm and SiLU, storing only the 4-bit input and recomputing the
 * intermediate values in the backward pass bounds the error more tightly
 * than caching quantised intermediates).  x_hat is the value
 * agoq_laaq_dequantize gives (fp32); then, in fp32,
 *   silu:     out = x_hat / (1 + exp(-x_hat)), computed as x_hat sigma(x_hat)
 *             from exp(-|x_hat|) (no overflow)
 *   rmsnorm:  per row of d values, out = x_hat / sqrt(mean(x_hat^2) + eps)
 *             * gamma (the sum of squares taken with compensated fp32
 *             addition)
 * Results are within a few units in the last fp32 place of the exact
 * operator on x_hat (not bit-reproducible against another implementation:
 * exp and the order of the sum are the library's).
 *
 *  packed, scale, block, bits, out, out_is_bf16   as for agoq_laaq_dequantize
 *  n                    (silu) elements, n % block == 0
 *  rows, d              (rmsnorm) the tensor [rows][d]; d % block == 0
 *  gamma        in      (rmsnorm) fp32 [d], 16-byte aligned
 *  eps                  (rmsnorm) eps >= 0, finite; with eps = 0 a row of zeros
 *                       gives NaN (0 / 0), as the formula does
 */
taco_status agoq_laaq_dequantize_silu(const uint8_t *packed, const float *scale, int64_t n, int32_t block,
                                      int32_t bits, void *out, int32_t out_is_bf16, taco_stream_t stream);
taco_status agoq_laaq_dequantize_rmsnorm(const uint8_t *packed, const float *scale, int64_t rows, int64_t d,
                                         int32_t block, int32_t bits, const float *gamma, float eps, void *out,
                                         int32_t out_is_bf16, taco_stream_t stream);

/*
 * taco_e4m3_encode - the compressor's FP8 encoder on its own ([TACO] 2.A:
 * the E4M3 format of the codes; 2.B.2: codes are taken with saturation at
 * the largest finite value).  codes[i] = E4M3FN(x[i]): round to nearest,
 * ties to even; |x| >= 448 (including +-Inf) gives +-448 (0x7E / 0xFE); a
 * value that rounds to zero keeps its sign (0x00 / 0x80); NaN gives a NaN
 * code (0x7F / 0xFF).  This is the conversion that step (5) of
 * taco_compress applies to y * scale.
 *
 *  x        in   fp32 [n], 16-byte aligned
 *  n             n >= 0
 *  codes    out  uint8 [n], 16-byte aligned, not overlapping x
 */
taco_status taco_e4m3_encode(const float *x, int64_t n, uint8_t *codes, taco_stream_t stream);

/*
 * taco_gemm_compress - the GEMM that produces a tensor-parallel partial sum,
 * with the compressor fused into its epilogue ([AGoQ] 2.C: quantisation
 * fused into the adjacent GEMM kernel, the tensor cores doing the product
 * and the CUDA cores the quantisation; applied to the [TACO] 2.B.1-2.B.2
 * compressor).  Y = A B^T is accumulated in fp32 on the tensor cores
 * (tcgen05, bf16 operands), and each 128-element block of each row of Y is
 * compressed exactly as taco_compress compresses a block, from the fp32
 * accumulator values (no bf16 rounding of Y).  The codes and scalars have
 * taco_compress's layout for a [M][N] tensor.
 *
 *  a_bf16   in   bf16 [M][K] (the layer input), 16-byte aligned
 *  b_bf16   in   bf16 [N][K] (the weight as [out][in]), 16-byte aligned
 *  M, N, K       M % 128 == 0, N % 128 == 0, K % 64 == 0, K > 0,
 *                M / 128 <= 65535; other shapes return TACO_ERR_UNSUPPORTED
 *  block         128 (others return TACO_ERR_UNSUPPORTED)
 *  e_target, eps as for taco_compress
 *  codes    out  uint8 [M][N]
 *  alpha    out  fp32 [M][N / 128]
 *  scale    out  fp32 [M][N / 128]
 *  y_out    out  optional fp32 [M][N]: the uncompressed Y, as accumulated
 *                (NULL: not written)
 *  workspace     optional device scratch for the split tail (below), 256-byte
 *                aligned, not overlapping any other argument, all zero before
 *                its first use; of workspace_bytes bytes.  NULL, 0 bytes or
 *                fewer than taco_gemm_workspace_bytes() gives: no split.
 *
 * Split tail: the kernel runs one CTA per SM over 128 x 256 tiles of Y (128
 * x 128 when N % 256 != 0).  When the tiles do not fill whole rounds of SMs,
 * the tiles of the last, partial round are each cut along K into 2-4
 * pieces of at least 2048 (if K allows and it saves at least an eighth of
 * a round) spread over all SMs; the pieces' fp32 partial sums meet in the
 * workspace and are added in piece order (so the result is the same on
 * every run), then compressed.  A call leaves the workspace's counters at
 * zero again, except after a watchdog error (taco_device_error bit 5),
 * after which the caller zeroes it before reusing it.  One call at a time
 * per workspace: calls on different streams need their own.  The split
 * changes the order of the fp32 additions of Y, not the bound on its error.
 */
taco_status taco_gemm_compress(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                               int32_t block, float e_target, float eps, uint8_t *codes, float *alpha,
                               float *scale, float *y_out, void *workspace, uint64_t workspace_bytes,
                               taco_stream_t stream);

/*
 * agoq_gemm_accumulate - the GEMM that produces a weight gradient, with the
 * FP8 accumulation into the main gradient fused into its epilogue ([AGoQ]
 * 2.C: quantisation fused into the adjacent GEMM kernel; 2.B: the main
 * gradient is kept in FP8 and each micro-batch's gradient is added by
 * dequantising, adding in FP32 and requantising).  G = A B^T is accumulated
 * in fp32 on the tensor cores (bf16 operands), and for each 128-element block
 * of each row of G, in place:
 *     g = decode(main_codes) * main_scale + G       (FP32: one rounded
 *                                                    multiply, one rounded add)
 *     main_scale = max|g| / 448 (1 for an all-zero block),
 *     main_codes = E4M3(g * (448 / max|g|))
 * -- agoq_fp8_accumulate's arithmetic, with the fp32 GEMM result in place of
 * the bf16 gradient.  For a weight gradient dW = dY^T X, pass A = dY^T and
 * B = X^T, both K-major (K = the tokens).
 *
 *  a_bf16      in      bf16 [M][K], 16-byte aligned
 *  b_bf16      in      bf16 [N][K], 16-byte aligned
 *  M, N, K, block      as for taco_gemm_compress
 *  main_codes  in/out  uint8 [M][N] (E4M3; all zero with main_scale 1 is
 *                      the zero gradient)
 *  main_scale  in/out  fp32 [M][N / 128], dequantisation multipliers
 *  y_out       out     optional fp32 [M][N]: G as accumulated (NULL: not written)
 *  workspace, workspace_bytes  as for taco_gemm_compress (the split tail)
 */
taco_status agoq_gemm_accumulate(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                 int32_t block, uint8_t *main_codes, float *main_scale, float *y_out,
                                 void *workspace, uint64_t workspace_bytes, taco_stream_t stream);

/*
 * agoq_gemm_laaq_quantize - the GEMM that produces an activation, with
 * AGoQ's block-wise activation quantisation fused into its epilogue ([AGoQ]
 * 2.C: quantisation in the adjacent GEMM kernel; 2.A: activations stored
 * block-wise in 4 bits, or 5, 6 or 8).  Y = A B^T is accumulated in fp32 on
 * the tensor cores (bf16 operands), and each 128-element block of each row
 * of Y is quantised exactly as agoq_laaq_quantize quantises a block, from
 * the fp32 values (no bf16 rounding of Y): amax = max|y|, q = qmax / amax,
 * code = rint(y q), multiplier amax / qmax (1 for an all-zero block).  The
 * packed stream and the multipliers have agoq_laaq_quantize's layout for the
 * row-major [M][N] tensor, so agoq_laaq_dequantize reads them back.
 *
 *  a_bf16      in      bf16 [M][K], 16-byte aligned
 *  b_bf16      in      bf16 [N][K], 16-byte aligned
 *  M, N, K, block      as for taco_gemm_compress (block 128)
 *  bits                4, 5, 6 or 8 (others return TACO_ERR_UNSUPPORTED)
 *  packed      out     uint8 [M * N * bits / 8], 16-byte aligned
 *  scale       out     fp32 [M][N / 128]
 *  y_out       out     optional fp32 [M][N]: Y as accumulated (NULL: not written)
 *  workspace, workspace_bytes  as for taco_gemm_compress (the split tail)
 */
taco_status agoq_gemm_laaq_quantize(const void *a_bf16, const void *b_bf16, int64_t M, int64_t N, int64_t K,
                                    int32_t block, int32_t bits, uint8_t *packed, float *scale, float *y_out,
                                    void *workspace, uint64_t workspace_bytes, taco_stream_t stream);

/*
 * taco_gemm_workspace_bytes - the workspace that taco_gemm_compress,
 * agoq_gemm_accumulate and agoq_gemm_laaq_quantize take for their split
 * tail on an M x N x K product on the current device (it depends on the SM
 * count); 0 when the shape gets no split.  No counterpart in the pages: a property of this implementation.
 *
 *  bytes  out  the size; shapes as for taco_gemm_compress (M or N = 0: 0)
 */
taco_status taco_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, uint64_t *bytes);

/*
 * Host pipeline: the two-shot local path between HOST buffers, overlapped.
 * A run computes, for a pinned bf16 host tensor x_host [P][rows][d] (P
 * shards), decompress(reduce(compress(shard 0), ..., compress(shard P-1)))
 * into a pinned host tensor out_host [rows][d] (fp32, or bf16 when
 * out_is_bf16): the result of taco_compress, taco_reduce_shards and
 * taco_decompress on the same data ([TACO] 2.B.3, the reducing rank's local
 * path of the two-shot AllReduce, with the exchange left out).  The rows are
 * split into chunks; one chunk's host-to-device copy (a single 2-D copy that
 * gathers the chunk's rows of all P shards), its kernels and its
 * device-to-host copy run on three streams, overlapping the other chunks.
 *
 * taco_host_pipeline_create - creates the pipeline's three CUDA streams and
 * its events on the current device (the one exception to "the library
 * never allocates": no device memory, only these CUDA objects and a small
 * host object) and reports the device workspace a run needs.
 *  P               1 .. TACO_MAX_SHARDS
 *  rows, d, block  as for taco_compress; rows >= 1
 *  chunks          1 .. 64 (capped at rows); chunk sizes differ by at most
 *                  the last chunk being shorter
 *  pipe_out        out: the new pipeline (NULL on error)
 *  workspace_bytes out: bytes of device workspace per run
 *
 * taco_host_pipeline_run - enqueues one pass and returns.  workspace is a
 * device buffer of workspace_bytes, 256-byte aligned, owned by the caller
 * and reused by every run of this pipeline.  x_host and out_host should be
 * pinned (page-locked) host memory: pageable memory works but its copies do
 * not overlap.  The first run is ordered after the work already queued on
 * `stream`; a later run of the same pipeline overlaps the previous run
 * chunk by chunk (its copy into a chunk's workspace waits only until the
 * previous run has compressed that chunk, its decompress only until the
 * previous run has copied that chunk out).  Every run makes `stream` wait
 * for its last copy-out, so out_host is complete when `stream` reaches that
 * point.  Must be called on the device the pipeline was created on.  After
 * a TACO_ERR_CUDA return the pipeline should be destroyed.
 *
 * taco_host_pipeline_destroy - releases the streams and events; work
 * already enqueued completes.
 */
typedef struct taco_host_pipeline taco_host_pipeline;
taco_status taco_host_pipeline_create(int32_t P, int64_t rows, int64_t d, int32_t block, int32_t chunks,
                                      int32_t out_is_bf16, taco_host_pipeline **pipe_out,
                                      uint64_t *workspace_bytes);
taco_status taco_host_pipeline_run(taco_host_pipeline *pipe, const void *x_host_bf16, void *out_host,
                                   void *workspace, float e_target, float eps, taco_stream_t stream);
taco_status taco_host_pipeline_destroy(taco_host_pipeline *pipe);

/*
 * taco_two_shot_host_noalloc - the result of taco_host_pipeline_run (fp32
 * output), for callers that cannot allocate device memory.  The papers have
 * no counterpart: this is a way to call the same path, not a step of the
 * method.
 *
 * Some callers cannot call cudaMalloc or any allocator: code that runs
 * inside an allocator or memory-pool callback, in a section where an
 * allocation could block or fail (a real-time or signal-handling path), or
 * a host program whose device memory belongs to another component.  This
 * call takes no workspace and allocates nothing, and creates no stream or
 * event.  Its intermediate buffers live in one device array inside the
 * library, TACO_NOALLOC_SCRATCH_MIB MiB on every GPU that loads the
 * library, held until the process exits.  The rows are processed in chunks
 * that fit the array, one after another on `stream`: no overlap between
 * copies and kernels, so it is slower than the pipeline.
 *
 *  P, rows, d, block, e_target, eps   as for taco_host_pipeline_create/run
 *  x_host_bf16  in   host bf16 [P][rows][d], should be pinned
 *  out_host     out  host fp32 [rows][d], should be pinned
 *
 * Limits and behaviour:
 *  - One row of all P shards and its intermediates must fit the array:
 *    P * d * (3 + 8/block) + d * (5 + 8/block) bytes (plus alignment) at most
 *    TACO_NOALLOC_SCRATCH_MIB MiB; larger rows return TACO_ERR_UNSUPPORTED
 *    without launching anything.  Any number of rows is accepted.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream
 *    capture.
 *  - Every call on a device uses the same array, which keeps the previous
 *    call's contents; nothing in it needs to start at zero.  Calls whose
 *    work overlaps on the GPU (other streams, other threads) race on it:
 *    serialise them.
 *  - `stream` must belong to the current device (the array used is the
 *    current device's); a stream of another device returns
 *    TACO_ERR_INVALID_ARG with nothing enqueued.
 *  - On TACO_ERR_CUDA, the copies and kernels of the chunks before the
 *    failing one may already be enqueued on `stream`: out_host is then
 *    partly written and its contents are undefined until the stream has
 *    drained.
 */
#define TACO_NOALLOC_SCRATCH_MIB 64
taco_status taco_two_shot_host_noalloc(int32_t P, int64_t rows, int64_t d, int32_t block,
                                       const void *x_host_bf16, float *out_host, float e_target,
                                       float eps, taco_stream_t stream);

/*
 * taco_device_error - watchdog flags of the kernels on the current device.
 * Every in-kernel wait gives up after about a second and sets a bit here
 * (bit 0: compressor, bit 1: decompressor, bit 4: taco_watchdog_selftest,
 * bit 5: the GEMMs taco_gemm_compress, agoq_gemm_accumulate and
 * agoq_gemm_laaq_quantize).
 * Synchronises the device.  With clear != 0 the flags are reset to 0 after
 * reading.
 */
taco_status taco_device_error(uint32_t *flags_out, int32_t clear);

/*
 * taco_watchdog_selftest - checks the watchdog on this GPU.  Launches one
 * warp that waits, with the kernels' time-limited wait, on a barrier that
 * nothing completes.  After about a second the wait gives up, the kernel
 * sets bit 4 of the flags that taco_device_error reads, and returns; the
 * context stays usable.  Nothing faults and nothing hangs.
 */
taco_status taco_watchdog_selftest(taco_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TACO_H */
