// Shared-memory staging of a scattered tile into contiguous output runs.
//
// Compaction and the one-bit split know, per tile, where each surviving
// element goes: a contiguous run of the output starting at a global offset
// that the look-back supplies.  Elements are first written to shared memory
// at their tile-local rank; the block then copies each run to global memory
// with 128-bit stores on 16-byte-aligned output chunks (scalar stores only
// at the two ragged ends), so the scatter costs no more global transactions
// than a streaming copy.
#pragma once

#include "core.cuh"

namespace devscan {

// Staging buffer geometry for a tile of TILE words: readable chunk indices
// -1 .. TILE/4 + 2 (the copy below reads one chunk past each end of a run
// and masks what it does not need).
template <int TILE>
struct StageBuffer {
    static constexpr int kWords = TILE + 16;
    static constexpr int kLead = 4;   // words before index 0
    static constexpr int kMinChunk = -1;
    static constexpr int kMaxChunk = TILE / 4 + 2;
};

// Copy stage[s0, s0 + cnt) to out[g0, g0 + cnt), out 16-byte aligned; no
// element at or past `limit` (the output's length) is ever written.
// Thread i of the block handles output chunk (g0 / 4 + i) and steps by
// THREADS.  Shared element (s0 + e - g0) lands in out[e]; with
// W = s0 - (g0 mod 4) = 4 * cw + a (0 <= a < 4), output chunk q_begin + i
// takes words a .. 3 of shared chunk cw + i and words 0 .. a-1 of the chunk
// after it, which comes from the next lane by a shuffle.  The loop's trip
// count is the same for every thread, so full warps reach each shuffle.
template <int THREADS, int TILE>
__device__ __forceinline__ void write_run_aligned(uint32_t *__restrict__ out, size_t g0, unsigned cnt,
                                                  const uint32_t *stage, int s0, int tid, size_t limit)
{
    using B = StageBuffer<TILE>;
    if (cnt == 0) return;
    const int lane = tid & 31;
    const size_t q_begin = g0 >> 2;
    const size_t q_end = (g0 + cnt + 3) >> 2;
    const size_t e_end = (g0 + cnt < limit) ? g0 + cnt : limit;
    const int W = s0 - static_cast<int>(g0 & 3);
    const int a = W & 3;
    const int cw = (W - a) / 4;
    const uint4 *stage4 = reinterpret_cast<const uint4 *>(stage);
    for (size_t i0 = 0; q_begin + i0 < q_end; i0 += THREADS) {
        const size_t i = i0 + static_cast<size_t>(tid);
        const size_t q = q_begin + i;
        int c = cw + static_cast<int>(i);
        if (c < B::kMinChunk || c + 1 > B::kMaxChunk) c = B::kMinChunk;
        const uint4 lo = stage4[c];
        uint4 hi;
        hi.x = __shfl_down_sync(kFullMask, lo.x, 1);
        hi.y = __shfl_down_sync(kFullMask, lo.y, 1);
        hi.z = __shfl_down_sync(kFullMask, lo.z, 1);
        hi.w = __shfl_down_sync(kFullMask, lo.w, 1);
        if (lane == 31) hi = stage4[c + 1];
        if (q >= q_end) continue;
        uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        uint32_t v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // select word a + j without dynamic register indexing
            uint32_t sel = w[j];
            sel = (a == 1) ? w[j + 1] : sel;
            sel = (a == 2) ? w[j + 2] : sel;
            sel = (a == 3) ? w[j + 3] : sel;
            v[j] = sel;
        }
        const size_t e0 = q * 4;
        if (e0 >= g0 && e0 + 4 <= e_end) {
            st_stream(reinterpret_cast<uint4 *>(out) + q, make_uint4(v[0], v[1], v[2], v[3]));
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (e0 + j >= g0 && e0 + j < e_end) out[e0 + j] = v[j];
        }
    }
}

// Same copy for an output that is only 4-byte aligned.
template <int THREADS>
__device__ __forceinline__ void write_run_scalar(uint32_t *__restrict__ out, size_t g0, unsigned cnt,
                                                 const uint32_t *stage, int s0, int tid, size_t limit)
{
    for (unsigned e = tid; e < cnt; e += THREADS)
        if (g0 + e < limit) out[g0 + e] = stage[s0 + static_cast<int>(e)];
}

// Copy a run staged in phase with its destination: element i of the run sits
// at stage[(g0 & 3) + i] (stage 16-byte aligned) and goes to out[g0 + i], out
// 16-byte aligned.  Shared chunk k then maps to output chunk g0 / 4 + k, so
// every whole chunk is one 128-bit load and one 128-bit store.  The words of
// the two ragged end chunks (at most three each) take a thread each, threads
// 0-3 the head and 4-7 the tail, after the loop: no thread branches off
// inside it.  Elements at or past `limit` are never written.
template <int THREADS>
__device__ __forceinline__ void write_run_direct(uint32_t *__restrict__ out, size_t g0, unsigned cnt,
                                                 const uint32_t *stage, int tid, size_t limit)
{
    static_assert(THREADS >= 8, "threads 0-7 store the ragged ends");
    if (cnt == 0 || g0 >= limit) return;   // (a start past the end only follows a timed-out wait)
    const unsigned a = static_cast<unsigned>(g0 & 3);
    const size_t room = limit - (g0 - a);   // words of out from the first chunk's start
    const unsigned end = a + cnt;
    const unsigned stop = room < end ? static_cast<unsigned>(room) : end;   // words [a, stop) are written
    const unsigned kb = (a + 3) >> 2, ke = stop >> 2;                      // the whole chunks: [kb, ke)
    uint4 *dst = reinterpret_cast<uint4 *>(out) + (g0 >> 2);
    const uint4 *src = reinterpret_cast<const uint4 *>(stage);
    for (unsigned k = kb + tid; k < ke; k += THREADS) st_stream(dst + k, src[k]);
    const unsigned w = tid < 4 ? a + tid : max(4 * ke, 4 * kb) + (tid - 4);
    if (tid < 8 && w < stop && (tid >= 4 || w < 4 * kb)) reinterpret_cast<uint32_t *>(dst)[w] = stage[w];
}

// write_run_direct that also counts the run's keys whose bit `nb` is 0, by
// the PART-position output part they land in: c0 for the part of out[g0],
// c1 for the next one (a run of at most PART keys spans two parts at most).
// A 16-byte chunk of out never straddles two parts, so each chunk adds its
// count to one of the two.
template <int THREADS, int PART>
__device__ __forceinline__ void write_run_direct_count(uint32_t *__restrict__ out, size_t g0, unsigned cnt,
                                                       const uint32_t *stage, int tid, size_t limit, int nb,
                                                       uint32_t &c0, uint32_t &c1)
{
    static_assert(THREADS >= 8, "threads 0-7 store the ragged ends");
    if (cnt == 0 || g0 >= limit) return;
    const unsigned a = static_cast<unsigned>(g0 & 3);
    const size_t room = limit - (g0 - a);
    const unsigned end = a + cnt;
    const unsigned stop = room < end ? static_cast<unsigned>(room) : end;
    const unsigned kb = (a + 3) >> 2, ke = stop >> 2;
    // staged word w lands at g0 - a + w: the next part starts at word `next`
    static_assert(PART % 4 == 0 && (PART & (PART - 1)) == 0, "parts of whole chunks, a power of two");
    const unsigned next = PART - static_cast<unsigned>((g0 - a) & (PART - 1));
    uint4 *dst = reinterpret_cast<uint4 *>(out) + (g0 >> 2);
    const uint4 *src = reinterpret_cast<const uint4 *>(stage);
    const uint32_t sel = byte_sel(nb);
    const int nbb = nb & 7;
    for (unsigned k = kb + tid; k < ke; k += THREADS) {
        const uint4 v = src[k];
        st_stream(dst + k, v);
        const uint32_t z = 4u - ones_at_bit(v, sel, nbb);
        if (4 * k < next)
            c0 += z;
        else
            c1 += z;
    }
    const unsigned w = tid < 4 ? a + tid : max(4 * ke, 4 * kb) + (tid - 4);
    if (tid < 8 && w < stop && (tid >= 4 || w < 4 * kb)) {
        const uint32_t key = stage[w];
        reinterpret_cast<uint32_t *>(dst)[w] = key;
        const uint32_t z = ((key >> nb) & 1u) ^ 1u;
        if (w < next)
            c0 += z;
        else
            c1 += z;
    }
}

// write_run_scalar with the same count as write_run_direct_count.
template <int THREADS, int PART>
__device__ __forceinline__ void write_run_scalar_count(uint32_t *__restrict__ out, size_t g0, unsigned cnt,
                                                       const uint32_t *stage, int s0, int tid, size_t limit, int nb,
                                                       uint32_t &c0, uint32_t &c1)
{
    const size_t first_part = g0 / PART;
    for (unsigned e = tid; e < cnt; e += THREADS) {
        if (g0 + e >= limit) continue;
        const uint32_t k = stage[s0 + static_cast<int>(e)];
        out[g0 + e] = k;
        const uint32_t z = ((k >> nb) & 1u) ^ 1u;
        if ((g0 + e) / PART == first_part)
            c0 += z;
        else
            c1 += z;
    }
}

}  // namespace devscan
