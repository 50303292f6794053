// Multi-bit LSD radix sort of uint32 keys: 8-bit digits, 4 passes (sm_103a).
//
// geek-doc.cn "并行前缀和 scan ..." section 一: radix sort rounds take "one or
// several bits", and the core of each round is a scan; lpnh.cn "并行扫描"
// section 4.2: per-digit counts, a prefix over them, then the scatter.
//
// One pass over digit p (bits 8p .. 8p+7):
//   1. radix_hist_kernel: every tile of 8,192 keys counts its 256 digit
//      values and stores them digit-major: hist[d * tiles + tile] (two
//      persistent 1,024-thread blocks per SM walk the tiles);
//   2. an exclusive add-scan of that array (the library's own scan; at 2^26
//      keys it is 2M counts, which the L2-resident scan takes) turns it into
//      every (digit, tile) run's first output position: all keys of smaller
//      digits, plus the keys of digit d in earlier tiles;
//   3. radix_scatter_kernel: every tile ranks its keys stably by digit --
//      eight warps of 32 rows, each row 32 consecutive keys in input order,
//      the lanes with equal digits
//      grouped by eight ballots (three rows in four) or the hardware match
//      (every fourth row), one counter row per warp in shared memory --
//      stages the tile sorted by digit and writes each digit's keys as one
//      contiguous run.
// Traffic: 12 bytes per key per pass (count read, scatter read and write),
// 48 per key for the sort, against 260 for the 32 one-bit splits.
#include <algorithm>

#include "core.cuh"
#include "launch.h"

namespace devscan {

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortRows = 32;                          // rows of 32 keys per warp
constexpr int kSortTile = kSortThreads * kSortRows;    // 8,192 keys
constexpr int kSortBuckets = 1 << kRadixDigitBits;     // 256
static_assert(kSortThreads >= kSortBuckets, "a thread per digit in the per-tile digit scan");

__device__ __forceinline__ unsigned digit_of(uint32_t key, int shift) { return (key >> shift) & (kSortBuckets - 1); }

// Lanes whose 8-bit digit equals this lane's, built from one ballot per digit
// bit; `valid`: this row's lanes that hold a key.  The ballots keep the
// integer pipe busy and the hardware match instruction the shared-memory
// pipe, so the scatter ranks one row in four with the match and the rest with
// ballots (measured: all ballots 288 us, all matches 496 us, one in four
// matches 252 us for a 2^26-key pass).
__device__ __forceinline__ unsigned match_digit(unsigned d, unsigned valid)
{
    unsigned eq = valid;
#pragma unroll
    for (int b = 0; b < kRadixDigitBits; ++b) {
        const unsigned bit = (d >> b) & 1u;
        const unsigned set = __ballot_sync(kFullMask, bit);
        eq &= set ^ (bit - 1u);   // set where this lane's bit is 1, ~set where it is 0
    }
    return eq;
}

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// hist[d * tiles + tile] = number of keys of the tile whose digit is d.  The
// count does not depend on the order of the keys, so the loads are plain
// coalesced 128-bit loads.  The kernel is persistent: block b counts tiles b,
// b + G, b + 2G, ... (G blocks, two per SM), and the next tile's keys are
// loading while the current tile is counted.  Shared-memory atomics go to one
// row of 256 counters per four warps; two sets of rows alternate, so one
// barrier per tile separates a tile's counting from the write-out (and
// clearing) of the tile before it.  Measured at 2^26 keys: 51.5 us per pass
// against 61 us for two tiles per block without the prefetch.
constexpr int kHistThreads = 1024, kHistBlocksPerSm = 2;
constexpr int kHistVecs = kSortTile / kHistThreads / 4;   // 16-byte loads per thread per tile (2)
__global__ void __launch_bounds__(kHistThreads, kHistBlocksPerSm)
radix_hist_kernel(const uint32_t *__restrict__ keys, size_t n, int shift, unsigned tiles, uint32_t *__restrict__ hist,
                  bool aligned)
{
    constexpr int COPIES = kHistThreads / 32 / 4;
    __shared__ uint32_t s_h[2][COPIES][kSortBuckets];   // 16 KB
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < 2 * COPIES * kSortBuckets; i += kHistThreads) (&s_h[0][0][0])[i] = 0;
    const unsigned G = gridDim.x;
    // keys of the tile being counted (cur) and of the next one (nxt); zeros
    // for tiles that take the scalar path or do not exist
    uint4 cur[kHistVecs], nxt[kHistVecs];
    auto load = [&](unsigned t, uint4 (&r)[kHistVecs]) {
        const size_t base = static_cast<size_t>(t) * kSortTile;
        const bool vec = t < tiles && aligned && base + kSortTile <= n;
#pragma unroll
        for (int v = 0; v < kHistVecs; ++v)
            r[v] = vec ? __ldcs(reinterpret_cast<const uint4 *>(keys + base) + v * kHistThreads + tid)
                       : make_uint4(0u, 0u, 0u, 0u);
    };
    load(blockIdx.x, cur);
    __syncthreads();   // the counters are clear
    int buf = 0;
    for (unsigned t = blockIdx.x; t < tiles; t += G) {
        load(t + G, nxt);
        const size_t base = static_cast<size_t>(t) * kSortTile;
        uint32_t *h = s_h[buf][warp / 4];
        if (aligned && base + kSortTile <= n) {
#pragma unroll
            for (int v = 0; v < kHistVecs; ++v) {
                atomicAdd(&h[digit_of(cur[v].x, shift)], 1u);
                atomicAdd(&h[digit_of(cur[v].y, shift)], 1u);
                atomicAdd(&h[digit_of(cur[v].z, shift)], 1u);
                atomicAdd(&h[digit_of(cur[v].w, shift)], 1u);
            }
        } else {   // the ragged last tile, or keys that are not 16-byte aligned
            for (int v = 0; v < kHistVecs; ++v)
                for (int j = 0; j < 4; ++j) {
                    const size_t e = base + static_cast<size_t>(v * kHistThreads + tid) * 4 + j;
                    if (e < n) atomicAdd(&h[digit_of(keys[e], shift)], 1u);
                }
        }
#pragma unroll
        for (int v = 0; v < kHistVecs; ++v) cur[v] = nxt[v];
        __syncthreads();   // tile t counted; the other set was written out and cleared before this barrier
        if (tid < kSortBuckets) {
            uint32_t c = 0;
#pragma unroll
            for (int w = 0; w < COPIES; ++w) {
                c += s_h[buf][w][tid];
                s_h[buf][w][tid] = 0;
            }
            hist[static_cast<size_t>(tid) * tiles + t] = c;
        }
        buf ^= 1;
    }
}

// Exclusive scan of one value per thread over threads 0 .. 255 of the block
// (every thread must call it; the others pass 0); uses s_tmp[8].
__device__ __forceinline__ uint32_t excl_scan_256(uint32_t v, uint32_t *s_tmp, int tid)
{
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(kFullMask, inc, d);
        if (lane >= d) inc += u;
    }
    if (warp < kSortBuckets / 32 && lane == 31) s_tmp[warp] = inc;
    __syncthreads();
    uint32_t base = 0;
    if (warp < kSortBuckets / 32)
        for (int w = 0; w < warp; ++w) base += s_tmp[w];
    __syncthreads();
    return base + inc - v;
}

// Rows ranked with the hardware match instead of ballots: every fourth.
constexpr unsigned kMatchRows = 0x11111111u;

// keys_in -> keys_out by the digit at `shift`; run_start[d * tiles + tile]:
// the first output position of the tile's keys of digit d.  Block b sorts
// tile tile0 + b; FULL: every tile of the launch holds kSortTile keys (the
// ragged last tile gets a launch of its own), which drops the bounds checks.
// Eight warps of 32 rows each: the per-tile work on the warps' digit
// counters (clearing, the digit scan over the warps, the staging offsets)
// is half that of sixteen warps of 16 rows, and measured at 2^26 keys the
// sort takes 1.12 against 1.20 ms.  Three blocks per SM (80 registers) beat
// two blocks at 128 registers (1.21 ms).  Each ballot is combined as
// set ^ (bit - 1) rather than by a select, and two rows' ranks are packed by
// one byte permute: 1.08 against 1.12 ms, and no spills.
template <bool FULL>
__global__ void __launch_bounds__(kSortThreads, 3)
radix_scatter_kernel(const uint32_t *__restrict__ keys_in, uint32_t *__restrict__ keys_out, size_t n, int shift,
                     unsigned tiles, unsigned tile0, const uint32_t *__restrict__ run_start)
{
    // per-warp digit counters; then each (warp, digit)'s first staged position
    __shared__ uint32_t s_wcount[kSortWarps][kSortBuckets];   // 8 KB
    __shared__ uint32_t s_keys[kSortTile];                     // 32 KB: the tile sorted by digit
    __shared__ uint32_t s_delta[kSortBuckets];                 // output position - staged position, per digit
    __shared__ uint32_t s_tmp[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned tile = tile0 + blockIdx.x;
    const size_t base = static_cast<size_t>(tile) * kSortTile;
    const size_t wbase = base + static_cast<size_t>(warp) * (kSortRows * 32);
    const unsigned len = FULL ? kSortTile : static_cast<unsigned>(n - base < kSortTile ? n - base : kSortTile);

    for (int i = tid; i < kSortWarps * kSortBuckets; i += kSortThreads) (&s_wcount[0][0])[i] = 0;
    if (tid < kSortBuckets) s_delta[tid] = run_start[static_cast<size_t>(tid) * tiles + tile];   // the run's start
    // keys of this warp's kWarpKeys that exist (the last tile is ragged)
    constexpr unsigned kWarpKeys = kSortRows * 32;
    const unsigned wlen = FULL ? kWarpKeys
                               : (n > wbase ? static_cast<unsigned>(n - wbase < kWarpKeys ? n - wbase : kWarpKeys) : 0u);
    uint32_t key[kSortRows];
#pragma unroll
    for (int r = 0; r < kSortRows; ++r) {
        const unsigned i = static_cast<unsigned>(r * 32 + lane);
        key[r] = (FULL || i < wlen) ? __ldcs(keys_in + wbase + i) : 0u;
    }
    __syncthreads();

    // rank within the warp: row by row (input order), equal digits grouped;
    // two rows' ranks (below kWarpKeys) share a register's 16-bit halves
    uint32_t rank2[kSortRows / 2];
    const unsigned lt = lanemask_lt();
    uint32_t rank_even = 0;   // the even row's rank, until its odd partner's
#pragma unroll
    for (int r = 0; r < kSortRows; ++r) {
        const bool has = FULL || static_cast<unsigned>(r * 32 + lane) < wlen;
        const unsigned valid = FULL ? kFullMask : __ballot_sync(kFullMask, has);
        const unsigned d = digit_of(key[r], shift);
        const unsigned same = ((kMatchRows >> r) & 1u) ? (__match_any_sync(kFullMask, d) & valid) : match_digit(d, valid);
        const int leader = has ? __ffs(same) - 1 : lane;
        uint32_t before = 0;
        if (has && lane == leader) {
            before = s_wcount[warp][d];
            s_wcount[warp][d] = before + __popc(same);
        }
        before = __shfl_sync(kFullMask, before, leader);
        const uint32_t rank = before + __popc(same & lt);
        if (r & 1)
            rank2[r / 2] = __byte_perm(rank_even, rank, 0x5410);
        else
            rank_even = rank;
    }
    __syncthreads();

    // per digit (thread d): the tile's count, the digit's first staged
    // position, then every warp's first staged position for the digit (one
    // lookup per key below) and the output shift of the digit's run
    uint32_t count = 0;
    if (tid < kSortBuckets) {
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) count += s_wcount[w][tid];
    }
    const uint32_t start = excl_scan_256(tid < kSortBuckets ? count : 0u, s_tmp, tid);
    if (tid < kSortBuckets) {
        uint32_t at = start;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) {
            const uint32_t c = s_wcount[w][tid];
            s_wcount[w][tid] = at;
            at += c;
        }
        s_delta[tid] -= start;   // output start - staged start (wraps as an unsigned offset)
    }
    __syncthreads();

    // stage sorted by digit (stable: warp order, then row order, then lane)
#pragma unroll
    for (int r = 0; r < kSortRows; ++r) {
        if (FULL || static_cast<unsigned>(r * 32 + lane) < wlen) {
            const unsigned d = digit_of(key[r], shift);
            s_keys[s_wcount[warp][d] + ((rank2[r / 2] >> (16 * (r & 1))) & 0xffffu)] = key[r];
        }
    }
    __syncthreads();

    // each digit's keys as one run: staged key i of digit d goes to
    // i + (first output position - first staged position of d)
#pragma unroll 4
    for (unsigned i = tid; i < len; i += kSortThreads) {
        const uint32_t k = s_keys[i];
        const size_t dst = static_cast<uint32_t>(i + s_delta[digit_of(k, shift)]);
        // full tiles: the run starts come from counts of the whole input, so
        // every destination is below n; the ragged tile keeps the guard
        if (FULL || dst < n) __stcs(keys_out + dst, k);
    }
}

cudaError_t launch_radix_pass(const uint32_t *src, uint32_t *dst, size_t n, int pass, uint32_t *hist,
                              const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    const unsigned tiles = tiles_for(n, kSortTile);
    const int shift = kRadixDigitBits * pass;
    const bool aligned = reinterpret_cast<uintptr_t>(src) % 16 == 0;
    const unsigned hist_blocks = std::min(tiles, static_cast<unsigned>(kHistBlocksPerSm * ws.num_sms));
    radix_hist_kernel<<<hist_blocks, kHistThreads, 0, s>>>(src, n, shift, tiles, hist, aligned);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_scan(ElemType::U32, kOpAdd, false, hist, hist, static_cast<size_t>(tiles) * kSortBuckets,
                    reinterpret_cast<uintptr_t>(hist) % 16 == 0, kCarryDefault, ws, spin_limit, s);
    if (e != cudaSuccess) return e;
    const unsigned full = static_cast<unsigned>(n / kSortTile);
    if (full > 0) radix_scatter_kernel<true><<<full, kSortThreads, 0, s>>>(src, dst, n, shift, tiles, 0u, hist);
    if (full < tiles) radix_scatter_kernel<false><<<1, kSortThreads, 0, s>>>(src, dst, n, shift, tiles, full, hist);
    return cudaGetLastError();
}

size_t radix_hist_words(size_t n) { return static_cast<size_t>(tiles_for(n, kSortTile)) * kSortBuckets; }

}  // namespace devscan
