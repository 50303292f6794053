// Radix-sort one-bit split and the LSD radix sort built on it (sm_103a).
//
// geek-doc.cn "并行前缀和 scan ..." section 一 (radix sort): scan the "bit is
// 0" predicate to get each zero's slot; a one goes to (total zeros + its
// rank among the ones).  lpnh.cn "并行扫描" section 4.2: per-digit counts,
// a prefix over them, then the scatter.
//
// The split kernel needs the total zero count Z before it can place any
// one, and a single pass cannot know Z.  So a zero-count pass runs first;
// inside the sort the zero count of bit b + 1 is accumulated by pass b
// while it scatters (a stable permutation keeps every bit's count), so the
// sort reads the keys 33 times instead of 64.
#include <algorithm>
#include <atomic>

#include "core.cuh"
#include "grid_sync.cuh"
#include "launch.h"
#include "pipeline_l2.cuh"
#include "split_policy.cuh"
#include "stage.cuh"

namespace devscan {

// Grid-stride zero count of one bit; one atomic per warp.
template <int THREADS, bool ALIGNED>
__global__ void __launch_bounds__(THREADS)
count_zeros_kernel(const uint32_t *__restrict__ keys, size_t n, int bit, unsigned *zeros)
{
    const size_t gtid = static_cast<size_t>(blockIdx.x) * THREADS + threadIdx.x;
    const size_t stride = static_cast<size_t>(gridDim.x) * THREADS;
    unsigned c = 0;
    size_t scalar_from = 0;
    if (ALIGNED) {
        const size_t nvec = n / 4;
        const uint4 *k4 = reinterpret_cast<const uint4 *>(keys);
        size_t i = gtid;
        for (; i + 3 * stride < nvec; i += 4 * stride) {
            const uint4 a = ld_stream(k4 + i), b = ld_stream(k4 + i + stride);
            const uint4 d = ld_stream(k4 + i + 2 * stride), e = ld_stream(k4 + i + 3 * stride);
            c += zeros_of(a, bit) + zeros_of(b, bit) + zeros_of(d, bit) + zeros_of(e, bit);
        }
        for (; i < nvec; i += stride) c += zeros_of(ld_stream(k4 + i), bit);
        scalar_from = nvec * 4;
    }
    for (size_t e = scalar_from + gtid; e < n; e += stride) c += ((keys[e] >> bit) & 1u) ? 0u : 1u;
    c = __reduce_add_sync(kFullMask, c);
    if ((threadIdx.x & 31) == 0 && c != 0) atomicAdd(zeros, c);
}

template <int THREADS, int VECS, bool ALIGNED>
__global__ void __launch_bounds__(THREADS)
split_kernel(const uint32_t *__restrict__ keys, uint32_t *__restrict__ out, size_t n, int bit,
             const unsigned *__restrict__ zeros_total, unsigned *next_zeros, int next_bit, unsigned num_tiles,
             unsigned long long *status, DevState *st, unsigned capacity, unsigned spin_limit)
{
    constexpr int NWARPS = THREADS / 32;
    constexpr int WARP_ITEMS = 32 * 4 * VECS;
    constexpr int TILE = THREADS * 4 * VECS;
    using B = StageBuffer<TILE>;
    __shared__ __align__(16) uint32_t s_stage_raw[B::kWords];
    __shared__ unsigned s_warp[NWARPS];
    __shared__ unsigned s_next[NWARPS];
    __shared__ unsigned s_prefix;
    __shared__ unsigned s_tile;
    uint32_t *s_stage = s_stage_raw + B::kLead;
    const AddU32 op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) s_tile = atomicAdd(&st->ticket, 1u);
    __syncthreads();
    const unsigned tile = s_tile;
    if (tile >= num_tiles) return;   // never taken: each launch hands out exactly num_tiles tickets
    const size_t tile_base = static_cast<size_t>(tile) * TILE;
    const size_t warp_base = tile_base + static_cast<size_t>(warp) * WARP_ITEMS;
    const bool full = tile_base + TILE <= n;
    const unsigned tile_len = full ? TILE : static_cast<unsigned>(n - tile_base);

    uint32_t x[VECS][4];
    load_rows<uint32_t, VECS, ALIGNED>(keys, warp_base, n, lane, full, x, 0u);

    // zero masks of `bit` (bit k of zmask[r] set when element k of row r is
    // inside [0, n) and has the bit clear) and the next bit's zero count
    uint32_t zmask[VECS], t[VECS];
    unsigned nz = 0;
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        const size_t e = warp_base + static_cast<size_t>(r * 32 + lane) * 4;
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const bool valid = full || (e + k < n);
            if (valid && !((x[r][k] >> bit) & 1u)) m |= 1u << k;
            if (valid && !((x[r][k] >> next_bit) & 1u)) ++nz;
        }
        zmask[r] = m;
        t[r] = __popc(m);
    }
    uint32_t row_excl[VECS], warp_total;
    warp_scan_rows<AddU32, VECS>(op, t, lane, row_excl, warp_total);
    if (next_zeros != nullptr) nz = __reduce_add_sync(kFullMask, nz);
    if (lane == 0) {
        s_warp[warp] = warp_total;
        s_next[warp] = nz;
    }
    __syncthreads();
    uint32_t warp_excl, tile_zeros;
    block_scan_warps<AddU32, NWARPS>(op, s_warp, warp, lane, warp_excl, tile_zeros);

    unsigned tag = 0;
    if (warp == 0) {
        tag = __shfl_sync(kFullMask, lane == 0 ? read_tag(st) : 0u, 0);
        publish<AddU32>(status, tile, tag, tile == 0 ? kFlagInclusive : kFlagAggregate, tile_zeros, lane);
    }
    if (next_zeros != nullptr && warp == NWARPS - 1 && lane == 0) {
        unsigned sum = 0;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) sum += s_next[w];
        if (sum != 0) atomicAdd(next_zeros, sum);
    }

    // stage: zeros at their zero rank, ones after all of the tile's zeros
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        uint32_t zr = warp_excl + row_excl[r];
        const uint32_t li0 = static_cast<uint32_t>(warp * WARP_ITEMS + (r * 32 + lane) * 4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t li = li0 + k;
            if (li < tile_len) {
                if ((zmask[r] >> k) & 1u) {
                    s_stage[zr] = x[r][k];
                    ++zr;
                } else {
                    s_stage[tile_zeros + (li - zr)] = x[r][k];
                }
            }
        }
    }

    if (warp == 0) {
        uint32_t prefix = 0;
        if (tile != 0) {
            prefix = lookback<AddU32, kLookbackPerLane>(op, status, tile, tag, &st->error, spin_limit, lane);
            publish<AddU32>(status, tile, tag, kFlagInclusive, prefix + tile_zeros, lane);
        }
        if (lane == 0) s_prefix = prefix;
        if (tile == num_tiles - 1) finish_launch(st, status, num_tiles, capacity, lane);
    }
    __syncthreads();

    const size_t zeros_before = s_prefix;
    const size_t z_total = *zeros_total;
    const size_t ones_at = z_total + (tile_base - zeros_before);
    if (ALIGNED) {
        write_run_aligned<THREADS, TILE>(out, zeros_before, tile_zeros, s_stage, 0, tid, n);
        write_run_aligned<THREADS, TILE>(out, ones_at, tile_len - tile_zeros, s_stage,
                                         static_cast<int>(tile_zeros), tid, n);
    } else {
        write_run_scalar<THREADS>(out, zeros_before, tile_zeros, s_stage, 0, tid, n);
        write_run_scalar<THREADS>(out, ones_at, tile_len - tile_zeros, s_stage, static_cast<int>(tile_zeros),
                                  tid, n);
    }
}


using SplitPipe = SplitPolicy<16, 4, 4, 2, 3, 10, 1>;
constexpr unsigned kSplitWaitLimit = 1u << 18;
constexpr size_t kSplitPipelineMinN = size_t(1) << 19;

cudaError_t launch_count_zeros(const uint32_t *keys, size_t n, int bit, unsigned *zeros, const Workspace &ws,
                               cudaStream_t s)
{
    constexpr int THREADS = 256;
    const size_t want = (n + THREADS * 16 - 1) / (THREADS * 16);
    const unsigned grid = static_cast<unsigned>(std::max<size_t>(1, std::min<size_t>(want, 4 * ws.num_sms)));
    if (reinterpret_cast<uintptr_t>(keys) % 16 == 0)
        count_zeros_kernel<THREADS, true><<<grid, THREADS, 0, s>>>(keys, n, bit, zeros);
    else
        count_zeros_kernel<THREADS, false><<<grid, THREADS, 0, s>>>(keys, n, bit, zeros);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Two-launch split (a standalone split, which must count the zeros first
// anyway): one cooperative launch counts the zeros of every 512-key part,
// meets at a grid barrier and turns the counts into the parts' exclusive
// offsets and the total Z; then a warp per part ranks its keys and writes its
// zeros run at its offset and its ones run at Z + (keys before the part -
// its offset).  The same bytes as the count pass plus the pipelined split
// (12 per key), without a chain between tiles.
// ---------------------------------------------------------------------------
constexpr int kSplitPart = 512, kSplitCountThreads = 1024, kSplitWriteWarps = 8, kSplitCountBatch = 2;

// off[p]: zeros of bit `bit` in parts 0 .. p-1 (first the part's own count);
// *zeros = all zeros.  Block b takes parts [b * chunk, (b + 1) * chunk).
__global__ void __launch_bounds__(kSplitCountThreads, 1)
split_count_kernel(const uint32_t *__restrict__ keys, size_t n, int bit, unsigned parts, unsigned chunk,
                   uint32_t *__restrict__ off, uint32_t *__restrict__ block_sums, unsigned *__restrict__ zeros,
                   DevState *st, unsigned spin_limit)
{
    constexpr int NW = kSplitCountThreads / 32, B = kSplitCountBatch;
    __shared__ uint32_t s_w[NW];
    __shared__ uint32_t s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned p0 = blockIdx.x * chunk, p1 = p0 + chunk < parts ? p0 + chunk : parts;
    // phase 1: warp w takes parts p0 + w, p0 + w + NW, ..., B at a time;
    // lane L reads the part's 16-byte groups L, L + 32, L + 64, L + 96
    uint32_t mine = 0;
    for (unsigned pb = p0 + warp; pb < p1; pb += NW * B) {
        uint4 q[B][4];
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const unsigned p = pb + k * NW;
            if (p < p1 && static_cast<size_t>(p + 1) * kSplitPart <= n) {
                const uint4 *k4 = reinterpret_cast<const uint4 *>(keys + static_cast<size_t>(p) * kSplitPart);
#pragma unroll
                for (int g = 0; g < 4; ++g) q[k][g] = __ldcs(k4 + g * 32 + lane);
            }
        }
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const unsigned p = pb + k * NW;
            if (p >= p1) break;   // warp-uniform
            uint32_t z = 0;
            if (static_cast<size_t>(p + 1) * kSplitPart <= n) {
#pragma unroll
                for (int g = 0; g < 4; ++g) z += zeros_of(q[k][g], bit);
            } else {
                const size_t e0 = static_cast<size_t>(p) * kSplitPart;
                for (size_t e = e0 + lane; e < n && e < e0 + kSplitPart; e += 32) z += ((keys[e] >> bit) & 1u) ? 0u : 1u;
            }
            z = __reduce_add_sync(kFullMask, z);
            if (lane == 0) off[p] = z;
            mine += z;
        }
    }
    if (lane == 0) s_w[warp] = mine;
    __syncthreads();
    if (warp == 0) {
        const uint32_t v = __reduce_add_sync(kFullMask, s_w[lane]);
        if (lane == 0) block_sums[blockIdx.x] = v;
    }

    const bool ok = grid_barrier(st, gridDim.x, spin_limit);

    // phase 2: the counts become offsets in place, a block of parts at a time
    if (warp == 0) {
        uint32_t v = 0;
        if (ok)
            for (unsigned b = lane; b < blockIdx.x; b += 32) v += __ldcg(block_sums + b);
        v = __reduce_add_sync(kFullMask, v);
        if (lane == 0) s_carry = v;
    }
    __syncthreads();
    uint32_t carry = s_carry;
    for (unsigned base = p0; base < p1; base += kSplitCountThreads) {
        const unsigned p = base + tid;
        const uint32_t c = p < p1 ? off[p] : 0u;   // this thread's own part: read before it is overwritten
        // exclusive scan over the block
        uint32_t inc = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t u = __shfl_up_sync(kFullMask, inc, d);
            if (lane >= d) inc += u;
        }
        if (lane == 31) s_w[warp] = inc;
        __syncthreads();
        uint32_t w = s_w[lane], wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t u = __shfl_up_sync(kFullMask, wi, d);
            if (lane >= d) wi += u;
        }
        const uint32_t total = __shfl_sync(kFullMask, wi, NW - 1);
        const uint32_t excl = __shfl_sync(kFullMask, wi - w, warp) + inc - c;
        if (p < p1) off[p] = carry + excl;
        carry += total;
        __syncthreads();   // s_w is read before the next round writes it
    }
    if (blockIdx.x == gridDim.x - 1 && tid == 0) *zeros = carry;
    grid_depart(st, gridDim.x);
}

// Warp w of block b splits part b * kSplitWriteWarps + w.
template <bool OUT_ALIGNED>
__global__ void __launch_bounds__(kSplitWriteWarps * 32)
split_write_kernel(const uint32_t *__restrict__ keys, uint32_t *__restrict__ out, size_t n, int bit, unsigned parts,
                   const uint32_t *__restrict__ off, const unsigned *__restrict__ zeros)
{
    constexpr int kStage = kSplitPart + 12;   // the zeros, the ones from the next 16-byte boundary, a spare chunk
    __shared__ __align__(16) uint32_t s_stage[kSplitWriteWarps][kStage];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned p = blockIdx.x * kSplitWriteWarps + warp;
    if (p >= parts) return;   // the whole warp: no barrier follows
    const size_t b = static_cast<size_t>(p) * kSplitPart;
    const unsigned part_len = n - b < static_cast<size_t>(kSplitPart) ? static_cast<unsigned>(n - b) : kSplitPart;
    uint32_t x[4][4], zmask[4];
    if (part_len == static_cast<unsigned>(kSplitPart)) {
        const uint4 *k4 = reinterpret_cast<const uint4 *>(keys + b);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 u = __ldcs(k4 + q * 32 + lane);
            x[q][0] = u.x;
            x[q][1] = u.y;
            x[q][2] = u.z;
            x[q][3] = u.w;
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) m |= ((x[q][j] >> bit) & 1u) << j;
            zmask[q] = m ^ 0xfu;
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const unsigned i = static_cast<unsigned>((q * 32 + lane) * 4 + j);
                x[q][j] = i < part_len ? keys[b + i] : 0u;
                if (i < part_len && !((x[q][j] >> bit) & 1u)) m |= 1u << j;
            }
            zmask[q] = m;
        }
    }
    const size_t zeros_at = off[p];
    const size_t ones_at = static_cast<size_t>(*zeros) + (b - zeros_at);
    split_write_warp<4>(x, zmask, part_len, zeros_at, ones_at, lane, s_stage[warp], out, OUT_ALIGNED, n);
}

size_t split_part_words(size_t n) { return (n + kSplitPart - 1) / kSplitPart; }

cudaError_t launch_split_two_pass(const uint32_t *keys, uint32_t *out, size_t n, int bit, unsigned *zeros,
                                  uint32_t *part_words, const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    const unsigned parts = static_cast<unsigned>(split_part_words(n));
    unsigned blocks = static_cast<unsigned>(ws.num_sms);
    const unsigned need = (parts + 31) / 32;
    if (blocks > need) blocks = need;
    const unsigned chunk = (parts + blocks - 1) / blocks;
    blocks = (parts + chunk - 1) / chunk;
    uint32_t *sums = ws.tile_sums;
    DevState *st = ws.state;
    void *args[] = {const_cast<uint32_t **>(&keys), &n, &bit, const_cast<unsigned *>(&parts),
                    const_cast<unsigned *>(&chunk), &part_words, &sums, &zeros, &st, &spin_limit};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(&split_count_kernel), dim3(blocks),
                                                dim3(kSplitCountThreads), args, 0, s);
    if (e != cudaSuccess) return e;
    const unsigned wblocks = (parts + kSplitWriteWarps - 1) / kSplitWriteWarps;
    if (reinterpret_cast<uintptr_t>(out) % 16 == 0)
        split_write_kernel<true><<<wblocks, kSplitWriteWarps * 32, 0, s>>>(keys, out, n, bit, parts, part_words, zeros);
    else
        split_write_kernel<false><<<wblocks, kSplitWriteWarps * 32, 0, s>>>(keys, out, n, bit, parts, part_words, zeros);
    return cudaGetLastError();
}

cudaError_t launch_split(const uint32_t *keys, uint32_t *out, size_t n, int bit, const unsigned *zeros,
                         unsigned *next_zeros, int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    const int next_bit = (bit < 31) ? bit + 1 : 31;
    const bool out_aligned = reinterpret_cast<uintptr_t>(out) % 16 == 0;
    const bool pipelined = reinterpret_cast<uintptr_t>(keys) % 16 == 0 &&
                           (carry == kCarryPipelined || (carry != kCarryLookback && n >= kSplitPipelineMinN));
    if (pipelined) {
        using G = PipeShape<SplitPipe>;
        auto kernel = pipeline_l2_kernel<SplitPipe>;
        static std::atomic<unsigned long long> attribute_set{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const unsigned long long devbit = 1ull << (dev & 63);
        if ((attribute_set.load() & devbit) == 0) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(G::kSmemBytes));
            if (e != cudaSuccess) return e;
            attribute_set.fetch_or(devbit);
        }
        const unsigned tiles = tiles_for(n, SplitPipe::kTile);
        const unsigned grid = tiles < static_cast<unsigned>(ws.num_sms) ? tiles : static_cast<unsigned>(ws.num_sms);
        SplitPipe::Args args{keys, out, n, bit, zeros, next_zeros, next_bit, out_aligned};
        kernel<<<grid, G::kThreads, G::kSmemBytes, s>>>(args, tiles, ws.status, ws.state, ws.capacity, spin_limit,
                                                        kSplitWaitLimit);
        return cudaGetLastError();
    }
    constexpr int THREADS = kSplitThreads, VECS = kSplitVecs;
    const unsigned tiles = tiles_for(n, kSplitTile);
    const bool aligned = (reinterpret_cast<uintptr_t>(keys) % 16 == 0) && out_aligned;
    if (aligned)
        split_kernel<THREADS, VECS, true><<<tiles, THREADS, 0, s>>>(keys, out, n, bit, zeros, next_zeros, next_bit,
                                                                   tiles, ws.status, ws.state, ws.capacity,
                                                                   spin_limit);
    else
        split_kernel<THREADS, VECS, false><<<tiles, THREADS, 0, s>>>(keys, out, n, bit, zeros, next_zeros, next_bit,
                                                                    tiles, ws.status, ws.state, ws.capacity,
                                                                    spin_limit);
    return cudaGetLastError();
}

}  // namespace devscan
