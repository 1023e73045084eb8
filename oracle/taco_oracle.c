/*
 * CPU oracle for the TACO ASH+DS FP8 codec and the AGoQ FP8 gradient paths.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, scalar statement of
 * what the GPU library computes.  It shares no code, header, table or constant
 * generator with the CUDA library, and the library never calls it.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg use it.
 *
 * Sources (web summaries of the papers):
 *   [TACO] "TACO: Efficient Communication Compression of Intermediate Tensors
 *          for Scalable Tensor-Parallel LLM Training" (gist.science summary of
 *          arXiv 2604.24088).
 *            2.A    why FP8: the E4M3 format, exponent-spaced codes
 *            2.B.1  Adaptive Scale-Hadamard (ASH): per-block energy
 *                   normalisation, then an orthogonal Hadamard rotation
 *            2.B.2  Dual-Scale (DS) quantisation: pre-transform alpha_k,
 *                   post-transform s_k keeping values inside +-Q_max;
 *                   decompression inverts the process with both scales
 *            2.B.3  fused operator; two-shot AllReduce (ReduceScatter +
 *                   AllGather): the per-rank local reduce of P shards
 *   [AGoQ] "AGoQ: Activation and Gradient Quantization for Memory-Efficient
 *          Distributed Training of LLMs" (gist.science summary of arXiv
 *          2605.00539).
 *            2.B    QuanGrad local accumulation (dequantise the FP8 main
 *                   gradient, add the new micro-batch gradient, requantise)
 *                   and the precision-preserving all-reduce, step 2 (local
 *                   FP32 sum of the received FP8 shards, requantise)
 *
 * Readings where the pages are silent (all arithmetic in double unless noted):
 *   - alpha_k = sqrt(E_target / (mean(x^2) + eps)), stored as fp32.
 *   - Hadamard: Sylvester natural order, normalised by c = 1/sqrt(n).
 *   - s_k = fp32(Q_max / max|y|), Q_max = 448; an all-zero y gives s_k = 1;
 *     a quotient above FLT_MAX is clamped to FLT_MAX.
 *   - Codes: E4M3FN, round to nearest with ties to even, saturating at 448.
 *     The value handed to the encoder is rounded to fp32 first, so the code
 *     decision is taken in the precision the GPU takes it in.
 *   - Reduce: a sum (not a mean) of the dequantised shards, in shard order.
 *   - AGoQ arithmetic is FP32, the precision the AGoQ page gives for the
 *     all-reduce's local sum (and the one the accumulation is specified in):
 *     dequantise = one rounded fp32 multiply, sums are sequential fp32 adds
 *     in shard order, no fused multiply-add.  The stored per-block AGoQ
 *     scale is the dequantisation multiplier m = max|g| / 448 (1 for an
 *     all-zero block); codes are E4M3(g * q) with q = 448 / max|g|.
 *   - Build with -ffp-contract=off so that no compiler fuses a*b+c.
 *
 * Pins: every entry point is checked by the non-GPU tests against facts that
 * do not come from this file (E4M3 against torch's float8_e4m3fn and the
 * format definition; the transform against scipy's Sylvester matrix and
 * H*H = n*I; closed-form round trips; invariants; the quantisation error
 * bound).  No function here is "parity unpinned".
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_QMAX 448.0

/* ---------------------------------------------------------------- E4M3FN */
/* [TACO] 2.A: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 holds subnormals m * 2^-9; fields 1..15 hold
 * (1 + m/8) * 2^(e-7); field 15 with mantissa 7 is NaN; no infinities. */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest representable magnitude by a scan over all 127 non-negative finite
 * codes (0x00 .. 0x7E, ascending in value).  Ties go to the even code, i.e.
 * the code whose mantissa LSB is 0.  |v| >= 448 saturates to 0x7E.  The sign
 * bit of v is kept, so negative values that round to zero give 0x80. */
static double g_mag[127];
static int g_mag_ready = 0;

uint8_t oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    int best = 0, c;
    double best_d;
    if (!g_mag_ready) {
        for (c = 0; c < 127; ++c)
            g_mag[c] = oracle_e4m3_decode((uint8_t)c);
        g_mag_ready = 1;
    }
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    if (a >= ORACLE_QMAX)
        return (uint8_t)(sign | 0x7E);
    best_d = a;
    for (c = 1; c < 127; ++c) {
        double dist = fabs(a - g_mag[c]);
        if (dist < best_d || (dist == best_d && (c & 1) == 0)) {
            best = c;
            best_d = dist;
        }
    }
    return (uint8_t)(sign | best);
}

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------- Hadamard */
/* Unnormalised Walsh-Hadamard transform in Sylvester (natural) order:
 * for h = 1, 2, 4, ..., n/2 every pair (i, i+h) with bit h of i clear
 * becomes (a + b, a - b).  Equals multiplication by H_n with
 * H_1 = [1], H_2k = [[H_k, H_k], [H_k, -H_k]]. */
void oracle_fwht(double *v, int n)
{
    int h, i, j;
    for (h = 1; h < n; h <<= 1)
        for (i = 0; i < n; i += 2 * h)
            for (j = i; j < i + h; ++j) {
                double a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
}

static int valid_block(int n)
{
    return n >= 2 && n <= 4096 && (n & (n - 1)) == 0;
}

static float ds_scale(double maxabs)
{
    double q;
    if (maxabs == 0.0)
        return 1.0f;
    q = ORACLE_QMAX / maxabs;
    if (q > (double)FLT_MAX)
        return FLT_MAX;
    return (float)q;
}

/* One block of [TACO] 2.B.1-2.B.2, steps in the pages' order:
 *   1. energy      m = (1/n) sum x_i^2
 *   2. ASH scale   alpha = sqrt(E / (m + eps))   (kept as fp32 alpha_f)
 *   3. rotation    y = c * H_n (alpha_f * x)
 *   4. DS scale    s = Q_max / max|y|            (kept as fp32 s_f)
 *   5. codes       E4M3(y * s_f)
 * x and work are n doubles; work is scratch. */
static void compress_block(const double *x, int n, double e_target, double eps,
                           uint8_t *codes, float *alpha_out, float *scale_out, double *work)
{
    double m = 0.0, c = 1.0 / sqrt((double)n), maxabs = 0.0;
    float alpha_f, s_f;
    int i;
    for (i = 0; i < n; ++i)
        m += x[i] * x[i];
    m /= n;
    alpha_f = (float)sqrt(e_target / (m + eps));
    for (i = 0; i < n; ++i)
        work[i] = (double)alpha_f * x[i];
    oracle_fwht(work, n);
    for (i = 0; i < n; ++i) {
        work[i] *= c;
        if (fabs(work[i]) > maxabs)
            maxabs = fabs(work[i]);
    }
    s_f = ds_scale(maxabs);
    for (i = 0; i < n; ++i)
        codes[i] = oracle_e4m3_encode((float)(work[i] * (double)s_f));
    *alpha_out = alpha_f;
    *scale_out = s_f;
}

/* [TACO] 2.B.2 reconstruction: x_hat = c * H_n(decode(code) / s) / alpha.
 * H_n is symmetric and H_n H_n = n I, so c H_n is its own inverse. */
static void decompress_block(const uint8_t *codes, float alpha_f, float s_f, int n, double *out)
{
    double c = 1.0 / sqrt((double)n);
    int i;
    for (i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(codes[i]) / (double)s_f;
    oracle_fwht(out, n);
    for (i = 0; i < n; ++i)
        out[i] = c * out[i] / (double)alpha_f;
}

static int shape_ok(int64_t rows, int64_t d, int block)
{
    return rows >= 0 && d > 0 && valid_block(block) && d % block == 0;
}

/* Compress a bf16 tensor [rows, d]; blocks are contiguous runs of `block`
 * elements of the row-major tensor.  alpha and scale get rows*d/block fp32
 * values.  Returns 0, or -1 on a bad shape. */
int oracle_compress(const uint16_t *x_bf16, int64_t rows, int64_t d, int block,
                    float e_target, float eps, uint8_t *codes, float *alpha, float *scale)
{
    int64_t nb, k;
    int i;
    double *x, *work;
    if (!shape_ok(rows, d, block))
        return -1;
    nb = rows * d / block;
    x = (double *)malloc(sizeof(double) * block);
    work = (double *)malloc(sizeof(double) * block);
    for (k = 0; k < nb; ++k) {
        for (i = 0; i < block; ++i)
            x[i] = bf16_to_double(x_bf16[k * block + i]);
        compress_block(x, block, e_target, eps, codes + k * block, alpha + k, scale + k, work);
    }
    free(x);
    free(work);
    return 0;
}

/* Same as oracle_compress for a float64 input (used by the shard reduce). */
int oracle_compress_f64(const double *x, int64_t rows, int64_t d, int block,
                        float e_target, float eps, uint8_t *codes, float *alpha, float *scale)
{
    int64_t nb, k;
    double *work;
    if (!shape_ok(rows, d, block))
        return -1;
    nb = rows * d / block;
    work = (double *)malloc(sizeof(double) * block);
    for (k = 0; k < nb; ++k)
        compress_block(x + k * block, block, e_target, eps, codes + k * block, alpha + k,
                       scale + k, work);
    free(work);
    return 0;
}

/* Decompress into float64 (the GPU returns fp32; the double result is the
 * exact reconstruction it is compared against). */
int oracle_decompress(const uint8_t *codes, const float *alpha, const float *scale,
                      int64_t rows, int64_t d, int block, double *out)
{
    int64_t nb, k;
    if (!shape_ok(rows, d, block))
        return -1;
    nb = rows * d / block;
    for (k = 0; k < nb; ++k)
        decompress_block(codes + k * block, alpha[k], scale[k], block, out + k * block);
    return 0;
}

/* [TACO] 2.B.3 two-shot AllReduce, the local step on one rank, and [AGoQ]
 * 2.B step 2 (local sum in high precision): dequantise each of the P shards,
 * sum them in shard order 0..P-1, then compress the sum. */
int oracle_reduce_shards(int P, const uint8_t *const *codes, const float *const *alpha,
                         const float *const *scale, int64_t rows, int64_t d, int block,
                         float e_target, float eps, uint8_t *out_codes, float *out_alpha,
                         float *out_scale)
{
    int64_t nb, k;
    int p, i;
    double *sum, *one;
    if (!shape_ok(rows, d, block) || P < 1)
        return -1;
    nb = rows * d / block;
    sum = (double *)malloc(sizeof(double) * block);
    one = (double *)malloc(sizeof(double) * block);
    for (k = 0; k < nb; ++k) {
        for (i = 0; i < block; ++i)
            sum[i] = 0.0;
        for (p = 0; p < P; ++p) {
            decompress_block(codes[p] + k * block, alpha[p][k], scale[p][k], block, one);
            for (i = 0; i < block; ++i)
                sum[i] += one[i];
        }
        compress_block(sum, block, e_target, eps, out_codes + k * block, out_alpha + k,
                       out_scale + k, one);
    }
    free(sum);
    free(one);
    return 0;
}

/* AGoQ requantisation of one block of fp32 values: q = 448 / max|g| for the
 * codes, m = max|g| / 448 stored for dequantisation (both fp32 divisions). */
static void agoq_requantise(const float *g, int n, uint8_t *codes, float *scale_out)
{
    float amax = 0.0f, q = 1.0f, m = 1.0f;
    int i;
    for (i = 0; i < n; ++i)
        if (fabsf(g[i]) > amax)
            amax = fabsf(g[i]);
    if (amax > 0.0f) {
        q = 448.0f / amax;
        if (!(q <= FLT_MAX))
            q = FLT_MAX;
        m = amax / 448.0f;
    }
    for (i = 0; i < n; ++i) {
        const float v = g[i] * q;
        codes[i] = oracle_e4m3_encode(v);
    }
    *scale_out = m;
}

/* Dequantise one code to FP32: decode (exact) times the block multiplier. */
static float agoq_dequantise(uint8_t code, float m)
{
    const float d = (float)oracle_e4m3_decode(code);
    const float x = d * m;
    return x;
}

/* [AGoQ] 2.B local accumulation, in place: per block,
 *   g = dequantise(main) + grad      (FP32: one multiply, then one add)
 *   main' = requantise(g).
 * n must be a multiple of block. */
int oracle_agoq_accumulate(uint8_t *main_codes, float *main_scale, const uint16_t *grad_bf16,
                           int64_t n, int block)
{
    int64_t nb, k;
    int i;
    float *g;
    if (n < 0 || !valid_block(block) || n % block != 0)
        return -1;
    nb = n / block;
    g = (float *)malloc(sizeof(float) * block);
    for (k = 0; k < nb; ++k) {
        for (i = 0; i < block; ++i) {
            const float deq = agoq_dequantise(main_codes[k * block + i], main_scale[k]);
            const float grad = (float)bf16_to_double(grad_bf16[k * block + i]);
            g[i] = deq + grad;
        }
        agoq_requantise(g, block, main_codes + k * block, main_scale + k);
    }
    free(g);
    return 0;
}

/* The same accumulation step with an FP32 gradient, the form it takes when
 * it is fused into the GEMM that produces the gradient ([AGoQ] 2.C): the
 * GEMM's FP32 result is the value added, with no bf16 rounding. */
int oracle_agoq_accumulate_f32(uint8_t *main_codes, float *main_scale, const float *grad, int64_t n, int block)
{
    int64_t nb, k;
    int i;
    float *g;
    if (n < 0 || !valid_block(block) || n % block != 0)
        return -1;
    nb = n / block;
    g = (float *)malloc(sizeof(float) * block);
    for (k = 0; k < nb; ++k) {
        for (i = 0; i < block; ++i) {
            const float deq = agoq_dequantise(main_codes[k * block + i], main_scale[k]);
            g[i] = deq + grad[k * block + i];
        }
        agoq_requantise(g, block, main_codes + k * block, main_scale + k);
    }
    free(g);
    return 0;
}

/* [AGoQ] 2.B precision-preserving all-reduce, step 2: dequantise the P
 * received FP8 shards to FP32, sum them in FP32 in shard order, requantise. */
int oracle_agoq_reduce(int P, const uint8_t *const *codes, const float *const *scale, int64_t n,
                       int block, uint8_t *out_codes, float *out_scale)
{
    int64_t nb, k;
    int p, i;
    float *g;
    if (n < 0 || !valid_block(block) || n % block != 0 || P < 1)
        return -1;
    nb = n / block;
    g = (float *)malloc(sizeof(float) * block);
    for (k = 0; k < nb; ++k) {
        for (i = 0; i < block; ++i) {
            float sum = agoq_dequantise(codes[0][k * block + i], scale[0][k]);
            for (p = 1; p < P; ++p)
                sum = sum + agoq_dequantise(codes[p][k * block + i], scale[p][k]);
            g[i] = sum;
        }
        agoq_requantise(g, block, out_codes + k * block, out_scale + k);
    }
    free(g);
    return 0;
}

/* ------------------------------------------------------- INT8 ASH + DS */
/* [TACO] 5: the same ASH + DS pipeline with INT8 codes for hardware without
 * native FP8.  Steps 1-3 are those of compress_block; then
 *   4. s = fp32(127 / max|y|)   (1 for an all-zero y; clamped to FLT_MAX)
 *   5. code_i = round-to-nearest-even(fp32(y_i * s)), clamped to [-127, 127]
 * and the reconstruction is c * H(code / s) / alpha. */
static void compress_block_int8(const double *x, int n, double e_target, double eps, int8_t *codes,
                                float *alpha_out, float *scale_out, double *work)
{
    double m = 0.0, c = 1.0 / sqrt((double)n), maxabs = 0.0, q;
    float alpha_f, s_f = 1.0f;
    int i;
    for (i = 0; i < n; ++i)
        m += x[i] * x[i];
    m /= n;
    alpha_f = (float)sqrt(e_target / (m + eps));
    for (i = 0; i < n; ++i)
        work[i] = (double)alpha_f * x[i];
    oracle_fwht(work, n);
    for (i = 0; i < n; ++i) {
        work[i] *= c;
        if (fabs(work[i]) > maxabs)
            maxabs = fabs(work[i]);
    }
    if (maxabs > 0.0) {
        q = 127.0 / maxabs;
        s_f = q > (double)FLT_MAX ? FLT_MAX : (float)q;
    }
    for (i = 0; i < n; ++i) {
        const float v = (float)(work[i] * (double)s_f);
        double r = rint((double)v);
        if (r > 127.0)
            r = 127.0;
        if (r < -127.0)
            r = -127.0;
        codes[i] = (int8_t)r;
    }
    *alpha_out = alpha_f;
    *scale_out = s_f;
}

int oracle_compress_int8(const uint16_t *x_bf16, int64_t rows, int64_t d, int block, float e_target,
                         float eps, int8_t *codes, float *alpha, float *scale)
{
    int64_t nb, k;
    int i;
    double *x, *work;
    if (!shape_ok(rows, d, block))
        return -1;
    nb = rows * d / block;
    x = (double *)malloc(sizeof(double) * block);
    work = (double *)malloc(sizeof(double) * block);
    for (k = 0; k < nb; ++k) {
        for (i = 0; i < block; ++i)
            x[i] = bf16_to_double(x_bf16[k * block + i]);
        compress_block_int8(x, block, e_target, eps, codes + k * block, alpha + k, scale + k, work);
    }
    free(x);
    free(work);
    return 0;
}

int oracle_decompress_int8(const int8_t *codes, const float *alpha, const float *scale, int64_t rows,
                           int64_t d, int block, double *out)
{
    int64_t nb, k;
    int i;
    double c = 1.0 / sqrt((double)block);
    if (!shape_ok(rows, d, block))
        return -1;
    nb = rows * d / block;
    for (k = 0; k < nb; ++k) {
        double *o = out + k * block;
        for (i = 0; i < block; ++i)
            o[i] = (double)codes[k * block + i] / (double)scale[k];
        oracle_fwht(o, block);
        for (i = 0; i < block; ++i)
            o[i] = c * o[i] / (double)alpha[k];
    }
    return 0;
}

/* The uniform INT8 comparison point of [TACO] 2.A: per block of raw x, no
 * transform, q = clamp(rint(x * 127 / amax), -127, 127), x_hat = q * amax / 127
 * (an all-zero block reconstructs to zeros). */
int oracle_int8_roundtrip(const uint16_t *x_bf16, int64_t rows, int64_t d, int block, double *out)
{
    int64_t nb, k;
    int i;
    if (!shape_ok(rows, d, block))
        return -1;
    nb = rows * d / block;
    for (k = 0; k < nb; ++k) {
        double amax = 0.0;
        for (i = 0; i < block; ++i) {
            double v = fabs(bf16_to_double(x_bf16[k * block + i]));
            if (v > amax)
                amax = v;
        }
        for (i = 0; i < block; ++i) {
            double q = 0.0;
            if (amax > 0.0) {
                q = rint(bf16_to_double(x_bf16[k * block + i]) * 127.0 / amax);
                if (q > 127.0)
                    q = 127.0;
                if (q < -127.0)
                    q = -127.0;
            }
            out[k * block + i] = q * amax / 127.0;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ LAAQ */
/* [AGoQ] 2.A, layer-aware activation quantisation: the activations of the
 * layers that are quantised are stored block-wise in 4 bits (5, 6 or 8 bits
 * where the pipeline-stage bit-width compensation grants more memory).
 * Reading (the page gives no format): per block of `block` elements,
 *   amax  = max |x|
 *   qmax  = 2^(bits-1) - 1
 *   q     = fp32(qmax / amax)          (1 for an all-zero block)
 *   code  = clamp(round-to-nearest-even(fp32(x * q)), -qmax, qmax)
 *   m     = fp32(amax / qmax)          (1 for an all-zero block; stored)
 *   x_hat = fp32(code * m)
 * Codes are two's complement, packed into a little-endian bit stream:
 * element i occupies bits [i * bits, (i + 1) * bits) of the buffer, bit j of
 * the stream being bit (j % 8) of byte j / 8.  All arithmetic is fp32. */
static int laaq_args_ok(int64_t n, int block, int bits)
{
    return n >= 0 && (block == 32 || block == 64 || block == 128 || block == 256) && n % block == 0 &&
           (bits == 4 || bits == 5 || bits == 6 || bits == 8);
}

static void put_bits(uint8_t *stream, int64_t bitpos, uint32_t value, int bits)
{
    int j;
    for (j = 0; j < bits; ++j) {
        const int64_t b = bitpos + j;
        if ((value >> j) & 1u)
            stream[b / 8] |= (uint8_t)(1u << (b % 8));
        else
            stream[b / 8] &= (uint8_t)~(1u << (b % 8));
    }
}

static int32_t get_bits_signed(const uint8_t *stream, int64_t bitpos, int bits)
{
    uint32_t v = 0;
    int j;
    for (j = 0; j < bits; ++j) {
        const int64_t b = bitpos + j;
        v |= (uint32_t)((stream[b / 8] >> (b % 8)) & 1u) << j;
    }
    if (v & (1u << (bits - 1)))
        return (int32_t)v - (int32_t)(1u << bits);
    return (int32_t)v;
}

/* One block of fp32 values x[0 .. block) -> its codes at element offset
 * `first` of the stream, and its multiplier. */
static void laaq_quantize_block(const float *x, int block, int bits, uint8_t *packed, int64_t first,
                                float *scale)
{
    int i;
    const float qmax = (float)((1 << (bits - 1)) - 1);
    float amax = 0.0f, q = 1.0f, m = 1.0f;
    for (i = 0; i < block; ++i) {
        const float v = fabsf(x[i]);
        if (v > amax)
            amax = v;
    }
    if (amax > 0.0f) {
        q = qmax / amax;
        if (!(q <= FLT_MAX))
            q = FLT_MAX;
        m = amax / qmax;
    }
    for (i = 0; i < block; ++i) {
        const float v = x[i] * q;
        float r = rintf(v);
        if (r > qmax)
            r = qmax;
        if (r < -qmax)
            r = -qmax;
        put_bits(packed, (first + i) * (int64_t)bits, (uint32_t)(int32_t)r & ((1u << bits) - 1u), bits);
    }
    *scale = m;
}

int oracle_laaq_quantize(const uint16_t *x_bf16, int64_t n, int block, int bits, uint8_t *packed,
                         float *scale)
{
    int64_t nb, k;
    int i;
    float x[256];
    if (!laaq_args_ok(n, block, bits))
        return -1;
    nb = n / block;
    for (k = 0; k < nb; ++k) {
        for (i = 0; i < block; ++i)
            x[i] = (float)bf16_to_double(x_bf16[k * block + i]);  /* exact */
        laaq_quantize_block(x, block, bits, packed, k * block, scale + k);
    }
    return 0;
}

/* The same quantisation of fp32 values: the form it takes when it is fused
 * into the GEMM that produces the activation ([AGoQ] 2.C: quantisation in
 * the adjacent GEMM kernel), which quantises its fp32 result with no bf16
 * rounding in between. */
int oracle_laaq_quantize_f32(const float *x, int64_t n, int block, int bits, uint8_t *packed, float *scale)
{
    int64_t nb, k;
    if (!laaq_args_ok(n, block, bits))
        return -1;
    nb = n / block;
    for (k = 0; k < nb; ++k)
        laaq_quantize_block(x + k * block, block, bits, packed, k * block, scale + k);
    return 0;
}

int oracle_laaq_dequantize(const uint8_t *packed, const float *scale, int64_t n, int block, int bits,
                           float *out)
{
    int64_t i;
    if (!laaq_args_ok(n, block, bits))
        return -1;
    for (i = 0; i < n; ++i) {
        const float c = (float)get_bits_signed(packed, i * (int64_t)bits, bits);
        out[i] = c * scale[i / block];
    }
    return 0;
}

/* [AGoQ] 2.A, recomputation instead of caching: for RMSNorm and SiLU, AGoQ
 * stores only the block-wise quantised input and recomputes the operator's
 * output from it in the backward pass (a tighter error bound than caching a
 * quantised output).  Reading (the page names the operators, not their
 * formulas): SiLU(x) = x / (1 + exp(-x)); RMSNorm of a row of d values,
 * y_i = x_i / sqrt(mean_j(x_j^2) + eps) * g_i.  The input x is the
 * dequantised fp32 value exactly as oracle_laaq_dequantize gives it; the
 * operator then runs in double. */
int oracle_laaq_dequantize_silu(const uint8_t *packed, const float *scale, int64_t n, int block, int bits,
                                double *out)
{
    int64_t i;
    if (!laaq_args_ok(n, block, bits))
        return -1;
    for (i = 0; i < n; ++i) {
        const double x = (double)((float)get_bits_signed(packed, i * (int64_t)bits, bits) * scale[i / block]);
        out[i] = x / (1.0 + exp(-x));
    }
    return 0;
}

int oracle_laaq_dequantize_rmsnorm(const uint8_t *packed, const float *scale, int64_t rows, int64_t d, int block,
                                   int bits, const float *gamma, double eps, double *out)
{
    int64_t r, j;
    if (rows < 0 || d <= 0 || d % block != 0 || !laaq_args_ok(rows * d, block, bits) || !(eps >= 0.0))
        return -1;
    for (r = 0; r < rows; ++r) {
        double ss = 0.0, inv;
        for (j = 0; j < d; ++j) {
            const int64_t i = r * d + j;
            const double x = (double)((float)get_bits_signed(packed, i * (int64_t)bits, bits) * scale[i / block]);
            out[i] = x;
            ss += x * x;
        }
        inv = 1.0 / sqrt(ss / (double)d + eps);
        for (j = 0; j < d; ++j)
            out[r * d + j] = out[r * d + j] * inv * (double)gamma[j];
    }
    return 0;
}
