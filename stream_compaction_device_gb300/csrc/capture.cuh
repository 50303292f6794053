// One-pass capture for the fused-predicate compaction (sm_103a).
#pragma once

#include "core.cuh"
#include "grid_sync.cuh"

namespace devscan {

// Keep mask of four int32 values against a threshold: bit j set when
// (int32) v_j > t.
__device__ __forceinline__ uint32_t greater_mask(uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3, int32_t t)
{
    return (static_cast<int32_t>(v0) > t ? 1u : 0u) | (static_cast<int32_t>(v1) > t ? 2u : 0u) |
           (static_cast<int32_t>(v2) > t ? 4u : 0u) | (static_cast<int32_t>(v3) > t ? 8u : 0u);
}

// ---------------------------------------------------------------------------
// Fused-predicate compaction in one pass while the kept values fit in shared
// memory (pgsm.cn "SIMT数据依赖与并行前缀和" section 3.3: an element adds 1 to
// the output count when it is kept, and the exclusive prefix of those counts
// is its output position).  Run by a cooperative launch, one block
// per SM (the caller's grid):
//   stream   every warp owns a contiguous range of its block's chunk and
//            reads it in rounds of 1,024 values (eight 128-bit loads per lane
//            in flight, allocating no L1 lines).  It ranks a round's kept
//            values with one warp scan of its eight rows' counts (packed into
//            the bytes of two words) and appends them, in order, to its own
//            region of shared memory;
//   barrier  the blocks' kept totals cross one grid barrier;
//   write    every block folds the totals of the blocks before it, and every
//            warp writes its region out as one contiguous run.
// HBM moves the values once and the kept values once: 4 n + 4 K bytes.  A warp
// gives up when its region would overflow or when it fills faster than its
// share allows (its kept count passes the region's size times the fraction of
// its range read, plus kCaptureSlack).  Every warp then stops at its next
// round, no block writes, and the caller -- the fused predicate's pipelined
// kernel, which runs this first -- goes on with the pipeline.  After a capture
// gives up, the stream's next kCaptureBackoff calls skip it (the outcome of
// the call before is always final when a launch starts, by stream order), so
// a run of dense calls pays one attempt in kCaptureBackoff + 1.
// The regions are the pipelined kernel's whole dynamic shared memory (about
// 194 KB: the SM's carveout stays at 196 KB, leaving 60 KB of L1 for the
// loads in flight; measured at 2^26 with 1% kept, 216 KB of regions and a
// 228 KB carveout took 60.0 us against 52.3 us with 192 KB).
// ---------------------------------------------------------------------------
constexpr unsigned kCaptureRound = 1024;      // values a warp reads per round
constexpr unsigned kCaptureSlack = 64;        // kept values a warp may run ahead of its share
constexpr unsigned kCaptureBackoff = 16;      // calls a stream skips the capture for after one gave up

// A 128-bit load that allocates no L1 line (the capture's shared memory
// leaves L1 small, and a line a load allocates holds L1 space until its data
// arrives; 4% faster at 216 KB of regions).
__device__ __forceinline__ uint4 ld_no_l1(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t byte_sum(uint32_t w) { return (w & 0xffu) + ((w >> 8) & 0xffu) + ((w >> 16) & 0xffu) + (w >> 24); }

// Returns true when the capture wrote the result (out, *count); false when it
// gave up, and then the caller does the compaction.  The caller checks the
// back-off first (capture_backoff) and calls this only when it is zero.  Every
// block of the grid returns the same unless a grid-barrier wait ran out (the
// error word then says so).  NW warps per block; s_kept: NW regions of CAP
// values; chunk: the elements of each block, a multiple of NW rounds.
template <int NW, unsigned CAP>
__device__ __forceinline__ bool capture_gt(const uint32_t *__restrict__ in, int32_t threshold,
                                           uint32_t *__restrict__ out, int32_t *__restrict__ count, size_t n,
                                           size_t chunk, uint32_t *__restrict__ block_sums, DevState *st,
                                           unsigned spin_limit, uint32_t *s_kept)
{
    __shared__ uint32_t s_wcnt[NW];
    __shared__ uint32_t s_base, s_total;
    __shared__ int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned blocks = gridDim.x;
    const size_t begin = static_cast<size_t>(blockIdx.x) * chunk;
    const size_t end = begin + chunk < n ? begin + chunk : n;
    const size_t wpart = chunk / NW;   // a multiple of kCaptureRound
    const size_t wb = begin + static_cast<size_t>(warp) * wpart;
    const size_t we = wb + wpart < end ? wb + wpart : (wb < end ? end : wb);   // [wb, we), maybe empty
    uint32_t *region = s_kept + static_cast<size_t>(warp) * CAP;
    const volatile unsigned *abort_flag = &st->capture_abort;
    uint32_t kept = 0;
    bool give_up = false;
    unsigned round = 0;
    // a round's values: rows r = 0 .. 7 of 128, lane L holding 4 L .. 4 L + 3
    auto load_round = [&](size_t s, uint4 (&q)[8]) {
        if (s + kCaptureRound <= we) {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(in + s);
#pragma unroll
            for (int r = 0; r < 8; ++r) q[r] = ld_no_l1(v4 + r * 32 + lane);
        } else {   // the input's ragged end
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                uint32_t v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const size_t e = s + static_cast<size_t>(r * 128 + lane * 4 + j);
                    v[j] = e < we ? in[e] : 0u;
                }
                q[r] = make_uint4(v[0], v[1], v[2], v[3]);
            }
        }
    };
    // ranks a round and appends its kept values; false: stop (this warp
    // gave up, or another warp did)
    auto take_round = [&](size_t s, const uint4 (&q)[8]) -> bool {
        const bool full = s + kCaptureRound <= we;
        // whether another warp gave up, read every fourth round
        const unsigned stop = (round & 3u) == 3u ? __shfl_sync(kFullMask, *abort_flag, 0) : 0u;
        uint32_t nib[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            uint32_t valid = 0xfu;
            if (!full) {
                const size_t e = s + static_cast<size_t>(r * 128 + lane * 4);
                valid = e >= we ? 0u : (we - e >= 4 ? 0xfu : (1u << (we - e)) - 1u);
            }
            nib[r] = greater_mask(q[r].x, q[r].y, q[r].z, q[r].w, threshold) & valid;
        }
        const uint32_t pa = __popc(nib[0]) | (__popc(nib[1]) << 8) | (__popc(nib[2]) << 16) | (__popc(nib[3]) << 24);
        const uint32_t pb = __popc(nib[4]) | (__popc(nib[5]) << 8) | (__popc(nib[6]) << 16) | (__popc(nib[7]) << 24);
        uint32_t ia = pa, ib = pb;   // a row keeps at most 128, so the bytes never carry
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t ua = __shfl_up_sync(kFullMask, ia, d), ub = __shfl_up_sync(kFullMask, ib, d);
            if (lane >= d) {
                ia += ua;
                ib += ub;
            }
        }
        const uint32_t ta = __shfl_sync(kFullMask, ia, 31), tb = __shfl_sync(kFullMask, ib, 31);
        const uint32_t xa = ia - pa, xb = ib - pb;
        const uint32_t round_total = byte_sum(ta) + byte_sum(tb);
        const size_t done = (full ? s + kCaptureRound : we) - wb;
        const uint32_t after = kept + round_total;
        const bool over = after > CAP || static_cast<uint64_t>(after) * wpart >
                                             static_cast<uint64_t>(CAP) * done + static_cast<uint64_t>(kCaptureSlack) * wpart;
        if (stop != 0u || over) {   // (warp-uniform)
            give_up = over;
            return false;
        }
        uint32_t at = kept;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint32_t ex = r < 4 ? xa : xb, tot = r < 4 ? ta : tb;
            const int sh = 8 * (r & 3);
            uint32_t rank = at + ((ex >> sh) & 0xffu);
            if (nib[r] & 1u) region[rank++] = q[r].x;
            if (nib[r] & 2u) region[rank++] = q[r].y;
            if (nib[r] & 4u) region[rank++] = q[r].z;
            if (nib[r] & 8u) region[rank] = q[r].w;
            at += (tot >> sh) & 0xffu;
        }
        kept = after;
        ++round;
        return true;
    };
    // (holding two rounds in registers, the next loading while this one is
    // taken, at 512 threads and 120 registers, measured the same)
    for (size_t s = wb; s < we; s += kCaptureRound) {
        uint4 q[8];
        load_round(s, q);
        if (!take_round(s, q)) break;
    }
    if (give_up && lane == 0) atomicOr(&st->capture_abort, 1u);
    if (lane == 0) s_wcnt[warp] = kept;
    __syncthreads();
    if (warp == 0) {
        const uint32_t v = __reduce_add_sync(kFullMask, lane < NW ? s_wcnt[lane] : 0u);
        if (lane == 0) {
            block_sums[blockIdx.x] = v;
            s_total = v;
        }
    }
    // grid barrier; a block stops waiting once any warp has given up
    __syncthreads();
    if (tid == 0) {
        __threadfence();   // the block's total (and its warps' give-up flags) before its arrival
        atomicAdd(&st->grid_arrive, 1u);
        int abort = 0;
        unsigned spins = 0;
        while (ld_acquire(&st->grid_arrive) < blocks) {
            if (ld_acquire(&st->capture_abort) != 0u) break;
            if (++spins >= spin_limit) {
                atomicOr(&st->error, kErrTimeout);
                abort = 1;
                break;
            }
            __nanosleep(spins < 64 ? 32 : 256);
        }
        s_abort = (abort || ld_acquire(&st->capture_abort) != 0u) ? 1 : 0;
    }
    __syncthreads();
    const bool abort = s_abort != 0;
    if (!abort) {
        if (warp == 0) {
            uint32_t v = 0;
            for (unsigned b = lane; b < blockIdx.x; b += 32) v += __ldcg(block_sums + b);
            v = __reduce_add_sync(kFullMask, v);
            if (lane == 0) s_base = v;
        }
        __syncthreads();
        const uint32_t wpre = __reduce_add_sync(kFullMask, lane < warp ? s_wcnt[lane] : 0u);
        const size_t g0 = static_cast<size_t>(s_base) + wpre;
        for (uint32_t i = lane; i < kept; i += 32) __stcs(out + g0 + i, region[i]);
        if (blockIdx.x == blocks - 1 && tid == 0) *count = static_cast<int32_t>(s_base + s_total);
    }
    // the last block to leave records the outcome and resets the flag and
    // the barrier's counters for the next launch on the stream
    __syncthreads();
    if (tid == 0 && atomicAdd(&st->grid_depart, 1u) == blocks - 1) {
        st->capture_wait = abort ? kCaptureBackoff : 0u;
        st->capture_abort = 0u;
        st->grid_arrive = 0u;
        st->grid_depart = 0u;
    }
    return !abort;
}

// The stream's back-off: capture attempts still to skip after one gave up.
// Every thread reads it (one word, so no barrier is needed for the block to
// agree).
__device__ __forceinline__ unsigned capture_backoff(const DevState *st)
{
    return *reinterpret_cast<const volatile unsigned *>(&st->capture_wait);
}

// A skipped attempt counts one off the back-off.  Called by one thread of
// every block, after that block's read of the back-off: the last block to
// arrive writes the new count and resets the arrival counter.
__device__ __forceinline__ void capture_skip_depart(DevState *st, unsigned backoff, unsigned blocks)
{
    if (atomicAdd(&st->grid_depart, 1u) == blocks - 1) {
        st->capture_wait = backoff - 1u;
        st->grid_depart = 0u;
    }
}

// The capture's chunk per block for a grid of `blocks`: whole rounds for
// every one of its nw warps.
inline size_t capture_chunk(size_t n, unsigned blocks, int nw)
{
    const size_t unit = static_cast<size_t>(nw) * kCaptureRound;
    const size_t units = (n + unit - 1) / unit;
    return ((units + blocks - 1) / blocks) * unit;
}

}  // namespace devscan
