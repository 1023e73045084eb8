// Inline-PTX helpers for the sm_103a kernels: shared-memory mbarriers with
// time-limited waits, TMA tensor copies, and FP8 E4M3 / bf16 conversions.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace taco {

// Every wait on another agent (TMA engine, producer warp) gives up after this
// many nanoseconds of %globaltimer, records a flag and lets the kernel exit.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------- programmatic dependent launch --
// A kernel launched with programmatic stream serialization may start before
// the previous kernel in its stream has finished; it must not touch that
// kernel's outputs before pdl_wait() returns (which waits for the previous
// grid to complete and its memory to be visible).  Without that launch
// attribute the instruction is a no-op.
//
// No kernel here triggers its dependents early (griddepcontrol.
// launch_dependents): a dependent grid is released when its predecessor
// completes.  Measured on GB300 in the back-to-back compress -> reduce ->
// decompress step at the GPT-6.7B size, an early trigger at the start of
// every kernel made the step slower: 122.1 us against 120.3 us with the
// 16-element shard reduce, and 132.7 us against 118.9 us with the
// 32-element one.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if
// it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

// ------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 cache policies (createpolicy) for data read or written exactly once.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D tiled TMA copies with an L2 cache policy: a store shared -> global
// (as tma_store_2d), and a load global -> shared whose bytes complete on the
// mbarrier `bar`.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap *map, int32_t x, int32_t y, uint32_t src,
                                                  uint64_t pol)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint"
                 " [%0, {%1, %2}], [%3], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y,
                                                 uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

// 2-D tiled store shared -> global (rows past the tensor end are clipped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int32_t x, int32_t y,
                                             uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until no bulk group of this thread is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------- shared loads --

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// ---------------------------------------------------------- global loads --

// 16-byte streaming load through the non-coherent path (data read once).
__device__ __forceinline__ uint4 ldg128_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The same with an L2 cache policy (policy_evict_first() for inputs that
// nothing reads again, so that they do not displace data the next kernel
// reads).
__device__ __forceinline__ uint4 ldg128_stream_hint(const void *p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ void stg128_stream(void *p, uint4 v)
{
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ------------------------------------------- separately rounded products --
// a * b + c with the product rounded before the sum, on two lanes of a
// float2.  __fmul_rn / __fadd_rn are never contracted into a fused
// multiply-add, so terms that cancel exactly give exactly zero and the
// result is that of the stated arithmetic.

__device__ __forceinline__ float2 mul2_rounded(float2 a, float2 b)
{
    return make_float2(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y));
}

__device__ __forceinline__ float2 add2_rounded(float2 a, float2 b)
{
    return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
}

// ----------------------------------------------------------- conversions --

// bf16 halves of a 32-bit word to fp32 (exact).
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> two E4M3FN codes, round to nearest even, saturating to +-448.
// The low byte of the result holds `lo`, the high byte `hi`.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 -> four E4M3FN codes packed little-endian into one word.
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float a, float b, float c, float d)
{
    return f32x2_to_e4m3x2(a, b) | (f32x2_to_e4m3x2(c, d) << 16);
}

// Two E4M3FN codes (low byte = first element) -> two fp32 values (exact:
// every E4M3 value is an fp16 value, and every fp16 value an fp32 one).
__device__ __forceinline__ void e4m3x2_to_f32x2(uint32_t two_codes, float &lo, float &hi)
{
    uint32_t h2;
    uint16_t in = static_cast<uint16_t>(two_codes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

// Two fp32 -> two bf16 (round to nearest even), low half = lo.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

} // namespace taco
