// sync.cuh -- bulk copies (TMA), mbarriers, L2 prefetch and bounded waits.
//
// Every wait in the library is bounded in wall time (%globaltimer): a wait that
// gives up raises the workspace error word and the kernel drains without further
// work, so a lost signal becomes an error status instead of a hung GPU.
#pragma once

#include <stdint.h>

namespace moe {

constexpr unsigned long long kWaitNs = 250ull * 1000 * 1000;  // 0.25 s per wait

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete; false if the
// wait ran out of time (`limit` ns) or `abort` (a CTA-wide error word) became
// non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, volatile int *abort,
                                          unsigned long long limit = kWaitNs) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_test(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > limit) return false;
    }
}

// Global -> shared bulk copy completing on `bar` (bytes and addresses multiples of 16).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Fire-and-forget prefetch of a 16-byte aligned range into L2.
__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One thread waits until *p >= target (bounded by `limit` ns); on expiry it
// raises *err.  Returns false on expiry or when another CTA already raised *err.
__device__ __forceinline__ bool spin_geq(const unsigned *p, unsigned target, unsigned *err,
                                         unsigned long long limit = kWaitNs) {
    if (ld_acquire_gpu(p) >= target) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (ld_acquire_gpu(p) >= target) return true;
        if (*(volatile unsigned *)err) return false;
        if (global_ns() - t0 > limit) {
            atomicExch(err, 1u);
            return false;
        }
        __nanosleep(64);
    }
}

// One thread waits until the cumulative counter *p has advanced by `delta`
// past `base` (modulo 2^32; bounded by `limit` ns, no sleep); on expiry it
// raises *err.  Returns false on expiry or when another CTA already raised *err.
__device__ __forceinline__ bool spin_reach(const unsigned *p, unsigned base, unsigned delta, unsigned *err,
                                           unsigned long long limit = kWaitNs) {
    if (ld_acquire_gpu(p) - base >= delta) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (ld_acquire_gpu(p) - base >= delta) return true;
        if (*(volatile unsigned *)err) return false;
        if (global_ns() - t0 > limit) {
            atomicExch(err, 1u);
            return false;
        }
    }
}

// Programmatic dependent launch: let the next kernel on the stream start early;
// wait until the previous one has completed and its memory is visible (both are
// no-ops when the launch did not ask for it).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Prefetch of the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_line_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Release/acquire fence at GPU scope: this thread's earlier writes become visible
// before its later ones (with a relaxed counter update after it: a release).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Named barrier over `threads` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Arrives at a named barrier without waiting for it.
__device__ __forceinline__ void named_arrive(int id, int threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace moe
