// Helpers of the kernels that fold their chunks, combine the chunk totals
// once, then finish with every chunk's offset known (sm_103a): loads whose
// lines L2 keeps for a second read, a block's stream of whole parts through a
// ring of bulk-copied shared-memory stages, a block-wide exclusive scan, the
// last-arriving block's scan of the block totals, a grid-wide barrier (every
// block of a cooperative launch is resident, so a counter in the stream's
// device state can gather them), and programmatic dependent launch.
#pragma once

#include <atomic>

#include "core.cuh"
#include "pipeline.cuh"

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

// The block streams parts [p0, p1) of `src` (PART_BYTES each, every one whole
// and inside the buffer, `src` 16-byte aligned) through NSTG shared-memory
// stages of SP parts: thread 0 issues one bulk copy per stage, warp w calls
// fn(part, its bytes in shared memory) for the stage's parts w, w + warps, ...
// and a stage is refilled once every warp is done with it, so NSTG - 1 copies
// stay in flight while a stage is read.  `ring` holds NSTG * SP * PART_BYTES
// bytes (16-byte aligned), `full` NSTG mbarriers.  Returns false when a wait
// ran out; the copies still in flight have then been waited for.
template <int PART_BYTES, int SP, int NSTG, typename Fn>
__device__ bool stream_parts(const uint8_t *src, unsigned p0, unsigned p1, uint8_t *ring, uint64_t *full,
                             unsigned wait_limit, Fn &&fn)
{
    static_assert(PART_BYTES % 16 == 0, "a bulk copy moves a multiple of 16 bytes");
    const int tid = threadIdx.x, warp = tid >> 5, warps = blockDim.x >> 5;
    const unsigned stages = p1 > p0 ? (p1 - p0 + SP - 1) / SP : 0u;
    if (tid == 0) {
        for (int s = 0; s < NSTG; ++s) mbar_init(&full[s], 1);
        mbar_init_fence();
    }
    __syncthreads();
    auto issue = [&](unsigned k) {
        const unsigned a = p0 + k * SP, m = p1 - a < SP ? p1 - a : SP;
        uint64_t *bar = &full[k % NSTG];
        mbar_arrive_expect_tx(bar, m * PART_BYTES);
        bulk_load(ring + static_cast<size_t>(k % NSTG) * SP * PART_BYTES, src + static_cast<size_t>(a) * PART_BYTES,
                  m * PART_BYTES, bar);
    };
    if (tid == 0)
        for (unsigned k = 0; k < NSTG && k < stages; ++k) issue(k);
    unsigned k = 0;
    bool ok = true;
    for (; k < stages; ++k) {
        const unsigned slot = k % NSTG;
        const bool landed = mbar_wait(&full[slot], (k / NSTG) & 1u, wait_limit);
        if (landed) {
            const unsigned a = p0 + k * SP, m = p1 - a < SP ? p1 - a : SP;
            const uint8_t *stage = ring + static_cast<size_t>(slot) * SP * PART_BYTES;
            for (unsigned j = warp; j < m; j += warps) fn(a + j, stage + j * PART_BYTES);
        }
        if (!__syncthreads_and(landed)) {   // every thread takes the same branch
            ok = false;
            break;
        }
        if (tid == 0 && k + NSTG < stages) issue(k + NSTG);
    }
    if (!ok && tid == 0)   // stages k .. k + NSTG - 1 may still be landing
        for (unsigned j = k; j < stages && j < k + NSTG; ++j) (void)mbar_wait(&full[j % NSTG], (j / NSTG) & 1u, wait_limit);
    __syncthreads();
    return ok;
}

// Exclusive add-scan of one value per thread over the block; `total` gets the
// block's sum.  s_w holds THREADS / 32 words; the caller separates two calls
// with a barrier.
template <int THREADS>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *s_w, int tid, uint32_t &total)
{
    constexpr int NW = THREADS / 32;
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(kFullMask, inc, d);
        if (lane >= d) inc += u;
    }
    if (lane == 31) s_w[warp] = inc;
    __syncthreads();
    uint32_t w = lane < NW ? s_w[lane] : 0u, wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(kFullMask, wi, d);
        if (lane >= d) wi += u;
    }
    total = __shfl_sync(kFullMask, wi, NW - 1);
    return __shfl_sync(kFullMask, wi - w, warp) + inc - v;
}

// Every block of the grid calls this once with its total (block-uniform).
// The last block to arrive writes carry[b] = totals of blocks 0 .. b-1 for
// every block b, resets the arrival counter for the next launch on the
// stream, and returns true with the grand total in `total`; the others
// return false.  Needs gridDim.x <= THREADS; s_w as for block_excl_scan,
// free on entry.
template <int THREADS>
__device__ bool last_block_carries(uint32_t block_total, uint32_t *block_sums, uint32_t *carry, DevState *st,
                                   uint32_t *s_w, uint32_t &total)
{
    __shared__ int s_last;
    const int tid = threadIdx.x;
    if (tid == 0) {
        block_sums[blockIdx.x] = block_total;
        __threadfence();   // the total before the arrival that counts it
        s_last = atomicAdd(&st->grid_arrive, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return false;
    __threadfence();
    const uint32_t v = tid < static_cast<int>(gridDim.x) ? __ldcg(block_sums + tid) : 0u;
    const uint32_t excl = block_excl_scan<THREADS>(v, s_w, tid, total);
    if (tid < static_cast<int>(gridDim.x)) carry[tid] = excl;
    if (tid == 0) st->grid_arrive = 0;
    return true;
}

// floor(p / d) for the part indices of a launch without a division
// sequence: (p * m) >> 40 with m = ceil(2^40 / d).  With m d = 2^40 + r,
// 0 <= r < d, the product's extra term p r / 2^40 stays below 1 when
// p d < 2^40, so the floor is exact; the host passes m = 0 (divide) when it
// cannot promise that for every part index p < parts, or when p m could
// overflow 64 bits.
struct ChunkDiv {
    unsigned d;
    unsigned long long m;
    __device__ __forceinline__ unsigned of(unsigned p) const
    {
        return m != 0 ? static_cast<unsigned>((static_cast<unsigned long long>(p) * m) >> 40) : p / d;
    }
};
inline ChunkDiv chunk_div(unsigned d, unsigned parts)
{
    ChunkDiv c;
    c.d = d;
    const unsigned long long pd = static_cast<unsigned long long>(parts) * d;
    const bool exact = pd < (1ull << 40) && static_cast<unsigned long long>(parts) < (static_cast<unsigned long long>(d) << 23);
    c.m = exact ? ((1ull << 40) + d - 1) / d : 0ull;
    return c;
}

// Programmatic dependent launch: a grid launched after this one with
// launch_dependent() may start once every block here has called
// allow_dependent_launch() (or exited); it waits in wait_primary_grid() until
// this grid has completed and its writes are visible.
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_primary_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// Host side: raise `kernel`'s dynamic shared-memory limit to `bytes`, once
// per device (`done` holds a bit per device).
inline cudaError_t allow_dynamic_smem(const void *kernel, int bytes, std::atomic<unsigned long long> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if ((done.load() & bit) == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit);
    }
    return cudaSuccess;
}

// Host side: launch `kernel` on `s` as a programmatic dependent of the grid
// before it (see allow_dependent_launch); without a wait_primary_grid() call
// first, the kernel must not read what that grid writes.  The kernel's
// pointers to such data carry no __restrict__: the wait orders memory
// accesses only through its "memory" clobber, and a load through a restrict
// pointer may be moved above it (seen on GB300: a write-launch variant that
// read the count launch's total through a restrict pointer right after the
// wait sometimes got an earlier call's total).
template <typename... Params, typename... Args>
cudaError_t launch_dependent_smem(void (*kernel)(Params...), unsigned grid, unsigned threads, size_t smem,
                                  cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), unsigned grid, unsigned threads, cudaStream_t s,
                             Args... args)
{
    return launch_dependent_smem(kernel, grid, threads, 0, s, args...);
}

}  // namespace devscan
