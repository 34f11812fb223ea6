// Device helpers for sm_103a: mbarriers with bounded waits, 1-D bulk copies
// (global -> shared, completion counted on an mbarrier), programmatic
// dependent launch controls, and the packed-arithmetic building blocks of the
// dequantising dot product.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace q4d {

// Error bits latched in the device error word.
enum : int { kErrTimeout = 1, kErrDeviceCheck = 2 };

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread until the phase
// completes or `hint_ns` elapses (no busy spinning that would steal issue
// slots from the warps doing the arithmetic).
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// latches kErrTimeout) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait_suspend(bar, parity, 1000000u)) return true;
        if (globaltimer() - t0 > kWaitLimitNs) {
            if (err) atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// 1-D bulk copy global -> shared; bytes multiple of 16, both addresses
// 16-byte aligned; completion decrements the mbarrier's tx count.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Same with an L2 eviction-priority hint (weights are streamed once).
__device__ __forceinline__ void bulk_g2s_evict_first(uint32_t dst, const void* src,
                                                     uint32_t bytes, uint32_t bar,
                                                     uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Tagged activation words: fp16 value in the low half, a 16-bit tag in the
// high half.  One 32-bit store publishes value and readiness together, so a
// reader polls the data itself (one memory round trip) instead of a flag and
// then the data.  Loads and stores are relaxed at GPU scope (coherent at L2).
__device__ __forceinline__ uint4 ld_relaxed_v4(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Programmatic dependent launch.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over `count` threads (multiple of 32).
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads; every
// thread gets the same result.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// (a & b) | c in one instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two products of the halves of `v` with the fp16 scale, plus fp32 c:
// lo = v.lo * s + c, hi = v.hi * s + c (exact fp16 products, one fp32 rounding).
__device__ __forceinline__ float2 fma_h2_s_f32(uint32_t v, uint16_t s, float c) {
    float lo, hi;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; fma.rn.f32.f16 %0, l, %3, %4; "
        "fma.rn.f32.f16 %1, h, %3, %4; }"
        : "=f"(lo), "=f"(hi)
        : "r"(v), "h"(s), "f"(c));
    return make_float2(lo, hi);
}

// Dequantise one word of 8 codes and accumulate against x pairs: the codes
// OR-ed into the mantissa of 1024.0 (nibbles 0, 2, 4, 6 as 1024+q) or 64.0
// (nibbles 1, 3, 5, 7 as 64+q), w = s*(1024+q) + (b - 1024 s) (or the 64
// form) by one fp16 x fp16 -> fp32 FMA each (the product is exact), and w*x
// accumulated in fp32 two at a time.  xa holds (x0, x4, x1, x5) and xb
// (x2, x6, x3, x7) of each of the M vectors; acc[m] gets the pairs' sums.
template <int M>
__device__ __forceinline__ void word_mac(uint32_t q, uint16_t sh, float c1024, float c64, const float4* xa,
                                         const float4* xb, float2* acc) {
    const uint32_t q8 = q >> 8;
    const uint32_t v0 = and_or(q, 0x000F000Fu, 0x64006400u);   // 1024+q0, 1024+q4
    const uint32_t v1 = and_or(q, 0x00F000F0u, 0x54005400u);   // 64+q1,   64+q5
    const uint32_t v2 = and_or(q8, 0x000F000Fu, 0x64006400u);  // 1024+q2, 1024+q6
    const uint32_t v3 = and_or(q8, 0x00F000F0u, 0x54005400u);  // 64+q3,   64+q7
    const float2 d0 = fma_h2_s_f32(v0, sh, c1024);             // w0, w4
    const float2 d1 = fma_h2_s_f32(v1, sh, c64);               // w1, w5
    const float2 d2 = fma_h2_s_f32(v2, sh, c1024);             // w2, w6
    const float2 d3 = fma_h2_s_f32(v3, sh, c64);               // w3, w7
#pragma unroll
    for (int m = 0; m < M; ++m) {
        acc[m] = __ffma2_rn(d0, make_float2(xa[m].x, xa[m].y), acc[m]);
        acc[m] = __ffma2_rn(d1, make_float2(xa[m].z, xa[m].w), acc[m]);
        acc[m] = __ffma2_rn(d2, make_float2(xb[m].x, xb[m].y), acc[m]);
        acc[m] = __ffma2_rn(d3, make_float2(xb[m].z, xb[m].w), acc[m]);
    }
}


}  // namespace q4d
