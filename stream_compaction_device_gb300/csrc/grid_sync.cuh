// Helpers of the cooperative launches (sm_103a): loads whose lines L2 keeps
// for a second read, and a grid-wide barrier -- every block of the grid is
// resident, so a counter in the stream's device state can gather them.  Used
// by the kernels that fold their chunks, meet once, then finish with every
// chunk's offset known.
#pragma once

#include "core.cuh"

namespace devscan {

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 128-bit load whose lines L2 keeps (evict_last).
__device__ __forceinline__ uint4 ld_keep(const uint4 *p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// All `blocks` blocks meet here.  Returns false (and records a timeout) when
// the wait runs out.
__device__ inline bool grid_barrier(DevState *st, unsigned blocks, unsigned spin_limit)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();   // this block's total before its arrival
        atomicAdd(&st->grid_arrive, 1u);
        int ok = 1;
        unsigned spins = 0;
        while (ld_acquire(&st->grid_arrive) < blocks) {
            if (++spins >= spin_limit) {
                atomicOr(&st->error, kErrTimeout);
                ok = 0;
                break;
            }
            __nanosleep(spins < 64 ? 32 : 256);
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// The last block to leave resets the counters for the next launch on the
// stream (which cannot start before this one has ended).
__device__ inline void grid_depart(DevState *st, unsigned blocks)
{
    if (threadIdx.x == 0 && atomicAdd(&st->grid_depart, 1u) == blocks - 1) {
        st->grid_arrive = 0;
        st->grid_depart = 0;
    }
}

}  // namespace devscan
