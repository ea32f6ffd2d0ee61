// bulk.cuh -- bulk asynchronous copies between global and shared memory
// (the non-tensor form of the Tensor Memory Accelerator, sm_90 and later)
// and the shared-memory barriers that track them, as hand-written PTX.
//
//  * bulk_load: one thread asks the copy engine for `bytes` contiguous bytes
//    of global memory into shared memory; the barrier's transaction count is
//    decremented as they land, so a waiter sees the whole row at once.
//  * bulk_store: the reverse, shared to global, tracked by bulk groups
//    (commit, then wait until at most N groups are still reading).
//
// Addresses and sizes of both must be multiples of 16 bytes.  Every wait on
// a barrier here is bounded by a deadline on the global nanosecond timer, so
// a copy that never completes becomes an error status instead of a hang.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t arrivals)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(arrivals) : "memory");
}

// Makes earlier shared-memory writes of this thread visible to the copy
// engine (the async proxy).
__device__ __forceinline__ void fence_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders barrier initialisation before any use of the barriers by other
// threads or by the copy engine.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also announces `bytes` more bytes of copy traffic for
// the barrier's current phase.
__device__ __forceinline__ void mbar_arrive_expect(uint64_t *bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// One plain arrival (release: this thread's earlier accesses happen before
// the phase completes for a waiter).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity to complete; false if
// the global timer passed `deadline` first.
__device__ __forceinline__ bool mbar_wait_until(uint64_t *bar, uint32_t parity, uint64_t deadline)
{
    while (!mbar_test(bar, parity))
        if (global_ns() > deadline) return false;
    return true;
}

// mbar_wait_until that also gives up as soon as *abort is non-zero.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity,
                                                   uint64_t deadline, const volatile int *abort)
{
    while (!mbar_test(bar, parity))
        if (*abort || global_ns() > deadline) return false;
    return true;
}

// Barrier `id` (1..15) over the first `count` threads that reach it; count a
// multiple of 32.  Lets a subset of the block synchronise while other warps
// run independently.
__device__ __forceinline__ void named_barrier(int id, int count)
{
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(dst_smem)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, const void *src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst), "r"(smem_addr(src_smem)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Until at most N committed groups still have to read their shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}

// Until every committed group has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

}  // namespace moe
