// Shared-memory pipeline primitives for sm_103a: mbarriers and 1-D bulk
// (TMA) copies from global to shared memory, all through inline PTX.
//
// A bulk copy moves `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global memory into this block's shared memory and signals
// completion on an mbarrier as transaction bytes.  Waits are bounded: every
// wait loop gives up after `limit` polls and reports it to its caller.
#pragma once

#include <cstdint>

namespace devscan {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the asynchronous (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// One bounded poll: the thread may be suspended for at most about
// kSuspendHintNs while the phase is still open.
constexpr unsigned kSuspendHintNs = 1000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return done != 0;
}

// Wait for the completion of the barrier phase with the given parity; false
// when `limit` polls (each at most about kSuspendHintNs) pass first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, unsigned limit)
{
    for (unsigned i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_global, unsigned bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_global), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Named barrier over `count` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_sync(unsigned id, unsigned count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads:
// every thread gets the same answer, so a decision taken after it is uniform.
__device__ __forceinline__ bool named_sync_and(unsigned id, unsigned count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<unsigned>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

}  // namespace devscan
