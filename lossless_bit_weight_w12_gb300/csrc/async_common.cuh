// async_common.cuh -- mbarrier primitives, shared-memory loads and named
// barriers, inline PTX.
//
// Every wait is bounded: it waits with try_wait (the hardware parks the warp
// until the phase completes, for at most kSuspendNs at a time) and gives up
// after the CTA's wait limit (kWaitLimitNs unless a launch asks for a
// shorter one) of wall time, or as soon as another thread of the CTA has
// given up, recording W12_ERR_TIMEOUT in the caller's error word.  No kernel
// of this library can spin forever.
#pragma once

#include <cstdint>

#include "../../include/w12.h"

namespace w12 {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Shared per-CTA wait state: the abort flag every bounded wait polls, and the
// wall-time limit of one wait.
struct WaitCtl {
    int abort;
    int pad;
    uint64_t limit_ns;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy before first use.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the warp is parked by the hardware
// until the phase completes or about `ns` nanoseconds have passed, instead
// of polling (a polling loop takes issue slots from the warps that work).
constexpr uint32_t kSuspendNs = 200000;  // 0.2 ms: an abort is seen within it

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// sets ctl->abort and *err) on timeout, or false at once if the CTA has
// already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, WaitCtl *ctl, int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    volatile int *abort = &ctl->abort;
    const uint64_t limit = ctl->limit_ns;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (*abort) return false;
        if (mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
        if (global_timer_ns() - t0 > limit) {
            *abort = 1;
            if (err) atomicCAS(err, 0, W12_ERR_TIMEOUT);  // the first error of a call wins
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used only to let copies or
// tensor-core operations that are already in flight finish before the CTA
// exits after a timeout).
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_sleep(bar, parity, kSuspendNs)) {
        if (global_timer_ns() - t0 > limit_ns) return;
    }
}

__device__ __forceinline__ bool aborted(const WaitCtl *ctl) {
    return *reinterpret_cast<const volatile int *>(&ctl->abort) != 0;
}

// L2 policy for data read exactly once (the weight planes).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}


__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(addr));
    return r;
}

// Barrier over the first `nthreads` threads of the CTA (named barrier 1).
__device__ __forceinline__ void named_sync(uint32_t nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

}  // namespace w12
