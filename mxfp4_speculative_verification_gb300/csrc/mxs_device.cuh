// Device-side building blocks shared by the sm_103a kernels of libmxs:
// mbarrier phases, TMA bulk copies, bounded waits, PDL controls and the
// hardware E2M1 / E8M0 conversions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mxs.h"

namespace mxs {

// A bounded wait gives up after this many nanoseconds of %globaltimer and
// reports MXS_DEV_TIMEOUT instead of spinning forever.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Writes of this thread to shared memory, made visible to the async proxy
// (tensor-core and TMA reads that follow).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void report(int32_t* status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// sets MXS_DEV_TIMEOUT) if it has not completed within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) {
            report(status, MXS_DEV_TIMEOUT);
            return false;
        }
    }
}

// The same wait, letting the hardware suspend the thread (up to `hint_ns`
// per try) until the phase completes, so that a warp waiting a long time
// takes no issue slots from the warps it shares a scheduler with.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, int32_t* status,
                                                uint32_t hint_ns = 20000u) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, hint_ns)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            report(status, MXS_DEV_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------ bulk copies
// 1-D TMA copy global -> shared, completion counted on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ----------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------- format conversions
// Two E2M1 codes (one byte, element 2i in the low nibble) -> f16x2 with the
// low nibble in the low half.  Exact: every E2M1 value is an fp16 value.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low8) {
    uint32_t out;
    asm("{\n"
        " .reg .b8 lo, b1, b2, b3;\n"
        " mov.b32 {lo, b1, b2, b3}, %1;\n"
        " cvt.rn.f16x2.e2m1x2 %0, lo;\n"
        "}\n"
        : "=r"(out)
        : "r"(byte_in_low8));
    return out;
}

// The four bytes of a 32-bit word as four f16x2 (bytes 0..3 in order).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                  uint32_t& h2, uint32_t& h3) {
    asm("{\n"
        " .reg .b8 b0, b1, b2, b3;\n"
        " mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        " cvt.rn.f16x2.e2m1x2 %3, b3;\n"
        "}\n"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

// Two E8M0 scale bytes (low 16 bits: byte 0, byte 1) -> their exact values
// 2^(e-127) as fp32 (e = 0 gives the subnormal 2^-127, e = 255 gives NaN).
__device__ __forceinline__ void e8m0x2_to_f32x2(uint32_t two_bytes, float& s0, float& s1) {
    uint32_t bf2;
    asm("{\n"
        " .reg .b16 lo, hi;\n"
        " mov.b32 {lo, hi}, %1;\n"
        " cvt.rn.bf16x2.ue8m0x2 %0, lo;\n"
        "}\n"
        : "=r"(bf2)
        : "r"(two_bytes));
    s0 = __uint_as_float(bf2 << 16);
    s1 = __uint_as_float(bf2 & 0xFFFF0000u);
}

}  // namespace mxs
