// Multi-bit LSD radix sort of uint32 keys, 4-bit digits, 8 passes (sm_103a).
//
// geek-doc.cn "并行前缀和 scan ..." section 一: radix sort rounds take "one or
// several bits", and the core of each round is a scan; lpnh.cn "并行扫描"
// section 4.2: per-digit counts, a prefix over them, then the scatter.
//
// One pass over digit p (bits 4p .. 4p+3):
//   1. radix_hist_kernel: every tile of 4,096 keys counts its 16 digit
//      values and stores them digit-major: hist[d * tiles + tile];
//   2. an exclusive add-scan of that array (the library's own scan) turns it
//      into every (digit, tile) run's first output position: all keys of
//      smaller digits, plus the keys of digit d in earlier tiles;
//   3. radix_scatter_kernel: every tile ranks its keys stably by digit
//      (private per-thread digit counters in shared memory, then one block
//      scan over them in digit-major order), stages the tile sorted by digit
//      and writes its 16 runs, each contiguous in the output.
// Traffic: 12 bytes per key per pass (read, read, write) instead of the
// 8 bytes x 32 passes of the one-bit split sort.
#include "core.cuh"
#include "launch.h"

namespace devscan {

constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;   // keys per thread, contiguous (blocked layout)
constexpr int kSortTile = kSortThreads * kSortItems;   // 4,096
constexpr int kDigits = 16;

__device__ __forceinline__ unsigned digit_of(uint32_t key, int shift) { return (key >> shift) & 15u; }

// Blocked load: thread t takes keys [16 t, 16 t + 16) of the tile.  Keys past
// n are flagged invalid.
__device__ __forceinline__ void load_blocked(const uint32_t *__restrict__ keys, size_t base, size_t n, int tid,
                                             bool aligned, uint32_t (&k)[kSortItems])
{
    const size_t e0 = base + static_cast<size_t>(tid) * kSortItems;
    if (aligned && e0 + kSortItems <= n) {
        const uint4 *p = reinterpret_cast<const uint4 *>(keys + e0);
#pragma unroll
        for (int v = 0; v < kSortItems / 4; ++v) {
            const uint4 q = ld_stream(p + v);
            k[4 * v] = q.x;
            k[4 * v + 1] = q.y;
            k[4 * v + 2] = q.z;
            k[4 * v + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < kSortItems; ++j) k[j] = (e0 + j < n) ? keys[e0 + j] : 0u;
    }
}

// hist[d * tiles + tile] = number of keys of the tile whose digit is d.
__global__ void __launch_bounds__(kSortThreads)
radix_hist_kernel(const uint32_t *__restrict__ keys, size_t n, int shift, unsigned tiles, uint32_t *__restrict__ hist,
                  bool aligned)
{
    __shared__ unsigned s_count[kDigits];
    const int tid = threadIdx.x;
    const unsigned tile = blockIdx.x;
    if (tid < kDigits) s_count[tid] = 0;
    const size_t base = static_cast<size_t>(tile) * kSortTile;
    uint32_t k[kSortItems];
    load_blocked(keys, base, n, tid, aligned, k);
    // 16 digit counts packed as 16-bit fields of 8 words (a thread counts at
    // most 16 keys, a warp at most 512)
    uint32_t c[kDigits / 2];
#pragma unroll
    for (int w = 0; w < kDigits / 2; ++w) c[w] = 0;
    const size_t e0 = base + static_cast<size_t>(tid) * kSortItems;
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
        if (e0 + j < n) {
            const unsigned d = digit_of(k[j], shift);
            const uint32_t inc = 1u << ((d & 1u) * 16);
#pragma unroll
            for (int w = 0; w < kDigits / 2; ++w) c[w] += (d >> 1 == static_cast<unsigned>(w)) ? inc : 0u;
        }
    }
#pragma unroll
    for (int w = 0; w < kDigits / 2; ++w)
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) c[w] += __shfl_xor_sync(kFullMask, c[w], o);
    __syncthreads();
    if ((tid & 31) == 0) {
#pragma unroll
        for (int w = 0; w < kDigits / 2; ++w) {
            atomicAdd(&s_count[2 * w], c[w] & 0xffffu);
            atomicAdd(&s_count[2 * w + 1], c[w] >> 16);
        }
    }
    __syncthreads();
    if (tid < kDigits) hist[static_cast<size_t>(tid) * tiles + tile] = s_count[tid];
}

__global__ void __launch_bounds__(kSortThreads)
radix_scatter_kernel(const uint32_t *__restrict__ keys, uint32_t *__restrict__ out, size_t n, int shift,
                     unsigned tiles, const uint32_t *__restrict__ run_start, bool aligned)
{
    constexpr int NWARPS = kSortThreads / 32;
    // private digit counters: column tid of row d; scanned in place
    __shared__ uint32_t s_cnt[kDigits * kSortThreads];
    __shared__ uint32_t s_keys[kSortTile];
    __shared__ uint32_t s_warp[NWARPS];
    __shared__ uint32_t s_start[kDigits], s_tbase[kDigits + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned tile = blockIdx.x;
    const size_t base = static_cast<size_t>(tile) * kSortTile;
    const unsigned len = (n - base < static_cast<size_t>(kSortTile)) ? static_cast<unsigned>(n - base) : kSortTile;

#pragma unroll
    for (int d = 0; d < kDigits; ++d) s_cnt[d * kSortThreads + tid] = 0;
    if (tid < kDigits) s_start[tid] = run_start[static_cast<size_t>(tid) * tiles + tile];
    uint32_t k[kSortItems];
    unsigned long long loc = 0;   // 16 x 4-bit local offsets (each < 16)
    load_blocked(keys, base, n, tid, aligned, k);
    // local offset of each key among this thread's earlier keys of its digit
    // (a thread's own column: no other thread touches it)
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
        if (static_cast<unsigned>(tid * kSortItems + j) < len) {
            const unsigned d = digit_of(k[j], shift);
            const uint32_t o = s_cnt[d * kSortThreads + tid];
            s_cnt[d * kSortThreads + tid] = o + 1;
            loc |= static_cast<unsigned long long>(o) << (4 * j);
        }
    }
    __syncthreads();

    // exclusive scan of s_cnt in digit-major order: warp w scans words
    // [512 w, 512 w + 512) row by row (lane l reads word 32 r + l: no bank
    // conflicts), carrying the row totals; warp totals through shared memory
    {
        const int seg = warp * (kDigits * kSortThreads / NWARPS);
        uint32_t carry = 0;
#pragma unroll 4
        for (int r = 0; r < kDigits * kSortThreads / NWARPS / 32; ++r) {
            const uint32_t v = s_cnt[seg + 32 * r + lane];
            uint32_t inc = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t u = __shfl_up_sync(kFullMask, inc, d);
                if (lane >= d) inc += u;
            }
            s_cnt[seg + 32 * r + lane] = carry + inc - v;
            carry += __shfl_sync(kFullMask, inc, 31);
        }
        if (lane == 0) s_warp[warp] = carry;
    }
    __syncthreads();
    {
        uint32_t wex = 0;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) wex += (w < warp) ? s_warp[w] : 0u;
        const int seg = warp * (kDigits * kSortThreads / NWARPS);
        for (int r = 0; r < kDigits * kSortThreads / NWARPS / 32; ++r) s_cnt[seg + 32 * r + lane] += wex;
    }
    __syncthreads();
    if (tid <= kDigits) s_tbase[tid] = (tid < kDigits) ? s_cnt[tid * kSortThreads] : len;

    // stage the tile sorted by digit (stable: digit-major, then thread,
    // then a thread's own order)
#pragma unroll
    for (int j = 0; j < kSortItems; ++j) {
        if (static_cast<unsigned>(tid * kSortItems + j) < len) {
            const unsigned d = digit_of(k[j], shift);
            s_keys[s_cnt[d * kSortThreads + tid] + static_cast<uint32_t>((loc >> (4 * j)) & 15u)] = k[j];
        }
    }
    __syncthreads();

    // write the 16 runs: staged key i of digit d goes to
    // run_start[d, tile] + (i - first staged position of d)
    for (unsigned i = tid; i < len; i += kSortThreads) {
        const uint32_t key = s_keys[i];
        const unsigned d = digit_of(key, shift);
        const size_t dst = static_cast<size_t>(s_start[d]) + (i - s_tbase[d]);
        if (dst < n) out[dst] = key;
    }
}

cudaError_t launch_radix_pass(const uint32_t *src, uint32_t *dst, size_t n, int pass, uint32_t *hist,
                              const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    const unsigned tiles = tiles_for(n, kSortTile);
    const int shift = 4 * pass;
    const bool aligned = reinterpret_cast<uintptr_t>(src) % 16 == 0;
    radix_hist_kernel<<<tiles, kSortThreads, 0, s>>>(src, n, shift, tiles, hist, aligned);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_scan(ElemType::U32, kOpAdd, false, hist, hist, static_cast<size_t>(tiles) * kDigits,
                    reinterpret_cast<uintptr_t>(hist) % 16 == 0, kCarryDefault, ws, spin_limit, s);
    if (e != cudaSuccess) return e;
    radix_scatter_kernel<<<tiles, kSortThreads, 0, s>>>(src, dst, n, shift, tiles, hist, aligned);
    return cudaGetLastError();
}

size_t radix_hist_words(size_t n) { return static_cast<size_t>(tiles_for(n, kSortTile)) * kDigits; }

}  // namespace devscan
