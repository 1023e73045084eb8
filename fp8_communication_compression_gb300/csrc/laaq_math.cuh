// Quantisation arithmetic of AGoQ's block-wise activation codec (AGoQ,
// gist.science summary of arXiv 2605.00539, 2.A), shared by the stand-alone
// quantizer and the GEMM whose epilogue quantises its output (2.C).

#pragma once

#include <cfloat>
#include <cstdint>

namespace taco {

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

// The block's quantisation factors: q = qmax / amax (at most FLT_MAX) and
// the stored multiplier m = amax / qmax; q = m = 1 for a block of zeros.
template <int BITS> __device__ __forceinline__ void laaq_factors(float amax, float &q, float &m)
{
    constexpr float kQmax = static_cast<float>((1 << (BITS - 1)) - 1);
    q = 1.0f;
    m = 1.0f;
    if (amax > 0.0f) {
        q = fminf(kQmax / amax, FLT_MAX);
        m = amax / kQmax;
    }
}

}  // namespace taco
