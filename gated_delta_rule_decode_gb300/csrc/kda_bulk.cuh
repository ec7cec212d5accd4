// Bulk-copy (1-D TMA) and mbarrier helpers in inline PTX for sm_100+.
//
// Every wait is bounded: a wait that runs out of iterations returns false so
// the caller can record KDA_DEVERR_TIMEOUT instead of hanging the GPU.
//
// Two limits: kWaitLimit bounds the waits of a kernel's main path, and
// kDrainLimit bounds the waits that, after a main-path wait gave up, let the
// copies and products still in flight finish before the CTA releases its
// shared and tensor memory.  KDA_WAIT_LIMIT lowers the first one in a test
// build, so that the timeout path can be exercised without a stuck copy.
#pragma once

#include <stdint.h>

#ifndef KDA_WAIT_LIMIT
#define KDA_WAIT_LIMIT (1u << 22)
#endif

namespace kda {

constexpr uint32_t kWaitLimit = KDA_WAIT_LIMIT;  // main-path try_wait polls before giving up
constexpr uint32_t kDrainLimit = 1u << 22;       // polls of a drain wait

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes the initialised barrier visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// Non-suspending probe of phase `phase`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// Bounded wait on phase `phase`; false if the limit ran out.  A test build
// (KDA_WAIT_NONBLOCKING, with a small KDA_WAIT_LIMIT) polls without the
// hardware's suspend, so that the limit runs out on copies and products
// that are merely in flight and the timeout path can be exercised.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t phase) {
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
#ifdef KDA_WAIT_NONBLOCKING
        if (mbar_test_wait(bar, phase)) return true;
#else
        if (mbar_try_wait(bar, phase)) return true;
#endif
    }
    return false;
}

// Drain wait: phase `phase` must be the one of an operation that was issued
// and not yet observed complete (a wait on a phase that nothing will complete
// spins out the whole limit).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t phase) {
    for (uint32_t it = 0; it < kDrainLimit; ++it)
        if (mbar_try_wait(bar, phase)) return true;
    return false;
}

// Global -> shared bulk copy completing on `bar` (bytes: multiple of 16).
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Shared -> global bulk copy in the thread's bulk group.
__device__ __forceinline__ void bulk_s2g(void *dst_gmem, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}

// Hint: bring `bytes` (a multiple of 16) at a 16-byte aligned global address into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src_gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

// Global -> shared 2-D tensor load (box of the tensor map at (x, y)),
// completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst_smem, const void *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Shared -> global 2-D tensor store (box of the tensor map at (x, y)) in the
// thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const void *map, int x, int y, const void *src_smem) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_addr(src_smem))
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most one committed bulk group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_le1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Waits until every committed bulk group has completed (writes included).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Waits until the committed bulk stores have finished READING shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Orders this thread's earlier generic-proxy accesses to global memory before
// later async-proxy (bulk copy) accesses to the same locations.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace kda
