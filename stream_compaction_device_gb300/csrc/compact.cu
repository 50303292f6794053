// Stream compaction (sm_103a).
//
// geek-doc.cn "并行前缀和 scan ..." section 一 and lpnh.cn "并行扫描" section
// 4.1: each kept element's output slot is the exclusive add-scan of the 0/1
// predicate; pgsm.cn "SIMT数据依赖与并行前缀和" section 4.2: the two-kernel
// block-count variant and the last thread writing the total.  Three forms,
// chosen by size (measured): one tile per block with a look-back on kept
// counts (small inputs); the persistent two-pass pipeline (pipeline_l2.cuh
// with CompactPolicy) where the predicate scan, the carry, the staged scatter
// and the count happen in one launch; and, for large inputs with flags, two
// launches -- a count of 512-element parts with their offsets, then a warp
// per part writing its run -- which no tile chain slows down.
#include <atomic>

#include "core.cuh"
#include "grid_sync.cuh"
#include "launch.h"
#include "compact_policy.cuh"
#include "pipeline_l2.cuh"
#include "stage.cuh"

namespace devscan {

// GT: keep in[i] when (int32) in[i] > threshold (flags unused); otherwise
// keep it when flags[i] != 0.
template <int THREADS, int VECS, bool ALIGNED, bool OUT_ALIGNED, bool GT = false>
__global__ void __launch_bounds__(THREADS)
compact_kernel(const uint32_t *__restrict__ in, const uint8_t *__restrict__ flags, uint32_t *__restrict__ out,
               int32_t *__restrict__ count, size_t n, unsigned num_tiles, unsigned long long *status,
               DevState *st, unsigned capacity, unsigned spin_limit, int32_t threshold = 0)
{
    constexpr int NWARPS = THREADS / 32;
    constexpr int WARP_ITEMS = 32 * 4 * VECS;
    constexpr int TILE = THREADS * 4 * VECS;
    using B = StageBuffer<TILE>;
    __shared__ __align__(16) uint32_t s_stage_raw[B::kWords];
    __shared__ unsigned s_warp[NWARPS];
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

    uint32_t x[VECS][4];
    load_rows<uint32_t, VECS, ALIGNED>(in, warp_base, n, lane, full, x, 0u);
    uint32_t keep[VECS];
    if (GT) {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            const size_t e = warp_base + static_cast<size_t>(r * 32 + lane) * 4;
            uint32_t m = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if ((full || e + k < n) && static_cast<int32_t>(x[r][k]) > threshold) m |= 1u << k;
            keep[r] = m;
        }
    } else if (ALIGNED && full) {
        uint32_t f[VECS];
#pragma unroll
        for (int r = 0; r < VECS; ++r)
            f[r] = ld_stream_u32(reinterpret_cast<const uint32_t *>(flags + warp_base) + r * 32 + lane);
#pragma unroll
        for (int r = 0; r < VECS; ++r) keep[r] = nonzero_byte_mask(f[r]);
    } else {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            const size_t e = warp_base + static_cast<size_t>(r * 32 + lane) * 4;
            uint32_t m = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (e + k < n && flags[e + k] != 0) m |= 1u << k;
            keep[r] = m;
        }
    }

    uint32_t t[VECS];
#pragma unroll
    for (int r = 0; r < VECS; ++r) t[r] = __popc(keep[r]);
    uint32_t row_excl[VECS], warp_total;
    warp_scan_rows<AddU32, VECS>(op, t, lane, row_excl, warp_total);
    if (lane == 0) s_warp[warp] = warp_total;
    __syncthreads();
    uint32_t warp_excl, tile_total;
    block_scan_warps<AddU32, NWARPS>(op, s_warp, warp, lane, warp_excl, tile_total);

    unsigned tag = 0;
    if (warp == 0) {
        tag = __shfl_sync(kFullMask, lane == 0 ? read_tag(st) : 0u, 0);
        publish<AddU32>(status, tile, tag, tile == 0 ? kFlagInclusive : kFlagAggregate, tile_total, lane);
    }

    // stage the kept values at their tile-local rank
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        uint32_t rank = warp_excl + row_excl[r];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if ((keep[r] >> k) & 1u) {
                s_stage[rank] = x[r][k];
                ++rank;
            }
        }
    }

    if (warp == 0) {
        uint32_t prefix = 0;
        if (tile != 0) {
            prefix = lookback<AddU32, kLookbackPerLane>(op, status, tile, tag, &st->error, spin_limit, lane);
            publish<AddU32>(status, tile, tag, kFlagInclusive, prefix + tile_total, lane);
        }
        if (lane == 0) {
            s_prefix = prefix;
            if (tile == num_tiles - 1) *count = static_cast<int32_t>(prefix + tile_total);
        }
        if (tile == num_tiles - 1) finish_launch(st, status, num_tiles, capacity, lane);
    }
    __syncthreads();

    if (OUT_ALIGNED)
        write_run_aligned<THREADS, TILE>(out, s_prefix, tile_total, s_stage, 0, tid, n);
    else
        write_run_scalar<THREADS>(out, s_prefix, tile_total, s_stage, 0, tid, n);
}


// ---------------------------------------------------------------------------
// Two-launch compaction with flags (pgsm.cn "SIMT数据依赖与并行前缀和" section
// 4.2's count-then-scatter order, on parts of 512 elements):
//   compact_count_kernel  a block per SM streams its chunk of parts through
//                         shared memory: every part's keep mask (one bit per
//                         element, 64 bytes) and kept count, then the parts'
//                         offsets within the chunk; the last block to finish
//                         scans the chunk totals into chunk carries and
//                         writes *count;
//   compact_write_kernel  launched as a programmatic dependent of the count
//                         (its launch overlaps the count's tail): a warp per
//                         part takes its mask, ranks its kept elements,
//                         stages them and writes one run at the part's
//                         offset plus its chunk's carry; a part that keeps at
//                         most kSparseKept elements loads only the 16-byte
//                         groups of values that hold one.
// No part waits on another, so the write launch streams.  HBM moves the
// flags once, the masks (1/8 of the flags) twice, the values once (only
// their kept groups for sparse parts) and the kept values once.
// ---------------------------------------------------------------------------
constexpr int kPartElems = 512;
constexpr unsigned kSparseKept = 32;
constexpr int kCountThreads = 1024, kCountStageParts = 128, kCountStages = 3, kWriteWarps = 8, kWriteMinBlocks = 1;
constexpr int kWritePartsPerWarp = 4;
constexpr unsigned kCountWaitLimit = 1u << 18;
constexpr unsigned kMaxCountBlocks = 512;   // chunk totals and carries share the workspace's tile sums

// mask[16 p .. 16 p + 15] = part p's keep bits (bit i of word w: element
// 32 w + i); cnt[p] = its kept elements; off[p] = kept elements of the parts
// before p in its chunk.  Block b takes the chunk of parts [b * chunk,
// (b + 1) * chunk): its whole parts stream through NSTG shared-memory stages
// of SP parts (dynamic shared memory), the ragged last part of the input
// takes plain loads.  The last block writes carry[b] = kept elements of the
// chunks before b, and *count (block_sums: one word per block).
// The parts' offsets within the block's chunk [p0, p1), THREADS parts at a
// time: off[p] = counts of the chunk's parts before p.  Then the last block
// to arrive writes carry[b] = counts of the chunks before b for every block
// b, and *count.  Called by every thread of every block, after the block's
// counts are written.
template <int THREADS>
__device__ void chunk_offsets(const uint32_t *__restrict__ cnt, uint32_t *__restrict__ off, unsigned p0, unsigned p1,
                              uint32_t *__restrict__ block_sums, uint32_t *__restrict__ carry, int32_t *count,
                              DevState *st, uint32_t *s_w)
{
    const int tid = threadIdx.x;
    uint32_t run = 0;
    for (unsigned base = p0; base < p1; base += THREADS) {
        const unsigned p = base + tid;
        const uint32_t c = p < p1 ? cnt[p] : 0u;
        uint32_t total;
        const uint32_t excl = block_excl_scan<THREADS>(c, s_w, tid, total);
        if (p < p1) off[p] = run + excl;
        run += total;
        __syncthreads();   // s_w is read before the next round writes it
    }
    uint32_t all;
    if (last_block_carries<THREADS>(run, block_sums, carry, st, s_w, all) && tid == 0)
        *count = static_cast<int32_t>(all);
}

template <int THREADS, int SP, int NSTG>
__global__ void __launch_bounds__(THREADS, 1)
compact_count_kernel(const uint8_t *__restrict__ flags, size_t n, unsigned parts, unsigned chunk,
                     uint32_t *__restrict__ mask, uint32_t *__restrict__ cnt, uint32_t *__restrict__ off,
                     uint32_t *__restrict__ block_sums, uint32_t *__restrict__ carry, int32_t *__restrict__ count,
                     DevState *st)
{
    static_assert(THREADS >= static_cast<int>(kMaxCountBlocks), "the last block scans one chunk total per thread");
    constexpr int NW = THREADS / 32;
    extern __shared__ __align__(128) uint8_t s_ring[];
    __shared__ uint64_t s_full[NSTG];
    __shared__ uint32_t s_w[NW];
    allow_dependent_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned p0 = blockIdx.x * chunk, p1 = p0 + chunk < parts ? p0 + chunk : parts;
    const unsigned whole = static_cast<unsigned>(n / kPartElems);
    const unsigned q1 = p1 < whole ? p1 : (p0 > whole ? p0 : whole);   // [p0, q1): whole parts

    // phase 1: a part per warp; lane L takes flags 16 L .. 16 L + 15
    auto part_done = [&](unsigned p, uint32_t m16) {
        const uint32_t hi = __shfl_down_sync(kFullMask, m16, 1);
        if ((lane & 1) == 0) mask[static_cast<size_t>(p) * 16 + (lane >> 1)] = m16 | (hi << 16);
        const uint32_t c = __reduce_add_sync(kFullMask, static_cast<uint32_t>(__popc(m16)));
        if (lane == 0) cnt[p] = c;
    };
    const bool streamed = stream_parts<kPartElems, SP, NSTG>(
        flags, p0, q1, s_ring, s_full, kCountWaitLimit, [&](unsigned p, const uint8_t *part) {
            const uint4 q = reinterpret_cast<const uint4 *>(part)[lane];
            part_done(p, nonzero_byte_mask(q.x) | (nonzero_byte_mask(q.y) << 4) | (nonzero_byte_mask(q.z) << 8) |
                             (nonzero_byte_mask(q.w) << 12));
        });
    if (!streamed && tid == 0) atomicOr(&st->error, kErrTimeout);
    for (unsigned p = q1 + warp; p < p1; p += NW) {   // the input's ragged last part
        const size_t e = static_cast<size_t>(p) * kPartElems + 16u * lane;
        uint32_t m16 = 0;
        for (unsigned j = 0; j < 16; ++j)
            if (e + j < n && flags[e + j] != 0) m16 |= 1u << j;
        part_done(p, m16);
    }
    __syncthreads();   // every part's count written

    // phase 2: the parts' offsets within the chunk; the last block's carries
    chunk_offsets<THREADS>(cnt, off, p0, p1, block_sums, carry, count, st, s_w);
}

// The fused predicate's count launch: keep values[i] > threshold (signed).
// Block b takes the chunk of parts [b * chunk, (b + 1) * chunk); warp w takes
// its parts w, w + NW, ... two at a time, so each lane has eight 128-bit
// loads in flight (their lines marked to stay in L2, where the write launch's
// dense parts find them).  In a part, lane L reads the 16-byte chunks L,
// L + 32, L + 64 and L + 96: row q gives it the 4-bit keep mask of elements
// 128 q + 4 L .. + 3, which lies in the part's mask word 4 q + L / 8 at bit
// 4 (L % 8); an OR over the 8 lanes of each group gathers the word.
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
compact_gt_count_kernel(const uint32_t *__restrict__ in, int32_t threshold, size_t n, unsigned parts,
                        unsigned chunk, uint32_t *__restrict__ mask, uint32_t *__restrict__ cnt,
                        uint32_t *__restrict__ off, uint32_t *__restrict__ block_sums, uint32_t *__restrict__ carry,
                        int32_t *__restrict__ count, DevState *st)
{
    static_assert(THREADS >= static_cast<int>(kMaxCountBlocks), "the last block scans one chunk total per thread");
    constexpr int NW = THREADS / 32;
    __shared__ uint32_t s_w[NW];
    allow_dependent_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned p0 = blockIdx.x * chunk, p1 = p0 + chunk < parts ? p0 + chunk : parts;
    const unsigned whole = static_cast<unsigned>(n / kPartElems);
    const unsigned q1 = p1 < whole ? p1 : (p0 > whole ? p0 : whole);   // [p0, q1): whole parts
    const uint64_t keep_pol = policy_evict_last();

    auto load_part = [&](unsigned p, uint4 (&v)[4]) {
        const uint4 *v4 = reinterpret_cast<const uint4 *>(in + static_cast<size_t>(p) * kPartElems);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = ld_keep(v4 + q * 32 + lane, keep_pol);
    };
    auto nibbles = [&](const uint4 (&v)[4], uint32_t (&nib)[4]) {
#pragma unroll
        for (int q = 0; q < 4; ++q) nib[q] = greater_mask(v[q].x, v[q].y, v[q].z, v[q].w, threshold);
    };
    auto part_done = [&](unsigned p, const uint32_t (&nib)[4]) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w = nib[q] << (4 * (lane & 7));
            w |= __shfl_xor_sync(kFullMask, w, 1);
            w |= __shfl_xor_sync(kFullMask, w, 2);
            w |= __shfl_xor_sync(kFullMask, w, 4);
            if ((lane & 7) == 0) mask[static_cast<size_t>(p) * 16 + 4 * q + (lane >> 3)] = w;
        }
        const uint32_t c = __reduce_add_sync(
            kFullMask, static_cast<uint32_t>(__popc(nib[0] | (nib[1] << 4) | (nib[2] << 8) | (nib[3] << 12))));
        if (lane == 0) cnt[p] = c;
    };
    unsigned p = p0 + warp;
    for (; p + NW < q1; p += 2 * NW) {   // two whole parts per round
        uint4 a[4], b[4];
        load_part(p, a);
        load_part(p + NW, b);
        uint32_t na[4], nb[4];
        nibbles(a, na);
        nibbles(b, nb);
        part_done(p, na);
        part_done(p + NW, nb);
    }
    for (; p < q1; p += NW) {
        uint4 a[4];
        load_part(p, a);
        uint32_t na[4];
        nibbles(a, na);
        part_done(p, na);
    }
    for (p = q1 + warp; p < p1; p += NW) {   // the input's ragged last part
        const size_t base = static_cast<size_t>(p) * kPartElems;
        uint32_t na[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const size_t e = base + static_cast<size_t>((q * 32 + lane) * 4 + j);
                if (e < n && static_cast<int32_t>(in[e]) > threshold) m |= 1u << j;
            }
            na[q] = m;
        }
        part_done(p, na);
    }
    __syncthreads();   // every part's count written

    chunk_offsets<THREADS>(cnt, off, p0, p1, block_sums, carry, count, st, s_w);
}

// Warp w of block b writes the kWritePartsPerWarp consecutive parts from
// (b * kWriteWarps + w) * kWritePartsPerWarp.  Lanes 0 .. 15 take the 16 mask
// words of each part (bit i of word w: element 32 w + i), and each part's
// output offset is its offset within its chunk plus the chunk's carry.
//   - A part that keeps at most kSparseKept elements takes the sparse path:
//     its kept indices are listed in order in shared memory, lane i loads the
//     i-th kept value and stores it at the part's offset + i.  The loads of
//     all the warp's sparse parts are in flight together, so at low
//     selectivity a part costs one round trip to its values after its mask,
//     shared with the warp's other parts.
//   - A denser part loads all its values (lane L, row q: elements
//     128 q + 4 L .. + 3, whose keep bits are the nibble of mask word
//     4 q + L / 8), ranks them, stages them in phase with their destination
//     and writes one run (compact_write_warp); those parts go one after
//     another.
template <bool OUT_ALIGNED, int MIN_BLOCKS>
__global__ void __launch_bounds__(kWriteWarps * 32, MIN_BLOCKS)
compact_write_kernel(const uint32_t *__restrict__ in, uint32_t *__restrict__ out, size_t n, unsigned parts,
                     ChunkDiv chunk, const uint32_t *mask, const uint32_t *off, const uint32_t *carry)
{
    constexpr int PPW = kWritePartsPerWarp;
    __shared__ __align__(16) uint32_t s_stage[kWriteWarps][kPartElems + 4];
    __shared__ uint16_t s_list[kWriteWarps][PPW][kSparseKept];
    wait_primary_grid();   // the count launch's masks, offsets and carries
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned p0 = (blockIdx.x * kWriteWarps + warp) * PPW;
    if (p0 >= parts) return;   // the whole warp: no block barrier follows
    uint32_t word[PPW], o[PPW], c[PPW];
#pragma unroll
    for (int k = 0; k < PPW; ++k) {
        const unsigned p = p0 + k;
        word[k] = (p < parts && lane < 16) ? mask[static_cast<size_t>(p) * 16 + lane] : 0u;
        o[k] = p < parts ? off[p] + carry[chunk.of(p)] : 0u;
    }
    // counts, and the sparse parts' kept indices in order
#pragma unroll
    for (int k = 0; k < PPW; ++k) {
        const uint32_t pc = static_cast<uint32_t>(__popc(word[k]));
        c[k] = __reduce_add_sync(kFullMask, pc);
        if (c[k] != 0 && c[k] <= kSparseKept) {   // (warp-uniform)
            uint32_t r = pc;
#pragma unroll
            for (int d = 1; d < 16; d <<= 1) {
                const uint32_t u = __shfl_up_sync(kFullMask, r, d);
                if (lane >= d) r += u;
            }
            r -= pc;   // kept elements in the words before this lane's
            uint32_t w = word[k];
            while (w != 0) {
                s_list[warp][k][r++] = static_cast<uint16_t>(32 * lane + (__ffs(w) - 1));
                w &= w - 1;
            }
        }
    }
    __syncwarp();
    uint32_t v[PPW];
#pragma unroll
    for (int k = 0; k < PPW; ++k)
        if (c[k] <= kSparseKept && static_cast<uint32_t>(lane) < c[k])
            v[k] = __ldcs(in + static_cast<size_t>(p0 + k) * kPartElems + s_list[warp][k][lane]);
#pragma unroll
    for (int k = 0; k < PPW; ++k)
        if (c[k] <= kSparseKept && static_cast<uint32_t>(lane) < c[k]) out[static_cast<size_t>(o[k]) + lane] = v[k];
    // dense parts, one after another
#pragma unroll
    for (int k = 0; k < PPW; ++k) {
        if (c[k] <= kSparseKept) continue;   // (warp-uniform)
        uint32_t x[4][4], keep[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            keep[q] = (__shfl_sync(kFullMask, word[k], 4 * q + (lane >> 3)) >> (4 * (lane & 7))) & 0xfu;
        const size_t b = static_cast<size_t>(p0 + k) * kPartElems;
        if (b + kPartElems <= n) {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(in + b);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 u = __ldcs(v4 + q * 32 + lane);
                x[q][0] = u.x;
                x[q][1] = u.y;
                x[q][2] = u.z;
                x[q][3] = u.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    x[q][j] = ((keep[q] >> j) & 1u) ? in[b + static_cast<size_t>((q * 32 + lane) * 4 + j)] : 0u;
        }
        compact_write_warp<4>(x, keep, o[k], lane, s_stage[warp], out, OUT_ALIGNED, n);
    }
}

size_t compact_part_words(size_t n) { return 18 * ((n + kPartElems - 1) / kPartElems); }   // mask, count, offset

// Parts per chunk of the count launch: one chunk per SM (fewer for small
// inputs, at least a part per warp each), at most kMaxCountBlocks chunks.
inline unsigned count_chunk(unsigned parts, unsigned warps, int num_sms)
{
    unsigned blocks = static_cast<unsigned>(num_sms) < kMaxCountBlocks ? static_cast<unsigned>(num_sms) : kMaxCountBlocks;
    const unsigned need = (parts + warps - 1) / warps;
    if (blocks > need) blocks = need;
    return (parts + blocks - 1) / blocks;
}

// The count launch: THREADS per block, NSTG * SP * 512 bytes of stages.
// part_words: mask[16 parts] | cnt[parts] | off[parts]; the workspace's tile
// sums hold the chunk totals (first kMaxCountBlocks words) and carries (next).
template <int THREADS, int SP, int NSTG>
cudaError_t launch_compact_count(const uint8_t *flags, size_t n, uint32_t *part_words, int32_t *count,
                                 unsigned chunk, const Workspace &ws, cudaStream_t s)
{
    static std::atomic<unsigned long long> smem_set{0};
    constexpr int kSmem = NSTG * SP * kPartElems;
    auto kernel = compact_count_kernel<THREADS, SP, NSTG>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kernel), kSmem, smem_set);
    if (e != cudaSuccess) return e;
    const unsigned parts = static_cast<unsigned>((n + kPartElems - 1) / kPartElems);
    const unsigned blocks = (parts + chunk - 1) / chunk;
    uint32_t *mask = part_words, *cnt = part_words + static_cast<size_t>(parts) * 16, *off = cnt + parts;
    kernel<<<blocks, THREADS, kSmem, s>>>(flags, n, parts, chunk, mask, cnt, off, ws.tile_sums,
                                          ws.tile_sums + kMaxCountBlocks, count, ws.state);
    return cudaGetLastError();
}

// The fused predicate's count launch (the same layout of part_words).
cudaError_t launch_compact_gt_count(const uint32_t *in, int32_t threshold, size_t n, uint32_t *part_words,
                                    int32_t *count, unsigned chunk, const Workspace &ws, cudaStream_t s)
{
    const unsigned parts = static_cast<unsigned>((n + kPartElems - 1) / kPartElems);
    const unsigned blocks = (parts + chunk - 1) / chunk;
    uint32_t *mask = part_words, *cnt = part_words + static_cast<size_t>(parts) * 16, *off = cnt + parts;
    compact_gt_count_kernel<kCountThreads><<<blocks, kCountThreads, 0, s>>>(
        in, threshold, n, parts, chunk, mask, cnt, off, ws.tile_sums, ws.tile_sums + kMaxCountBlocks, count,
        ws.state);
    return cudaGetLastError();
}

// gt: keep in[i] > threshold (the count launch reads the values; flags unused)
cudaError_t launch_compact_two_pass(const uint32_t *in, const uint8_t *flags, uint32_t *out, int32_t *count,
                                    size_t n, bool out_aligned, uint32_t *part_words, const Workspace &ws,
                                    cudaStream_t s, bool gt = false, int32_t threshold = 0)
{
    const unsigned parts = static_cast<unsigned>((n + kPartElems - 1) / kPartElems);
    const unsigned chunk = count_chunk(parts, kCountThreads / 32, ws.num_sms);
    cudaError_t e = gt ? launch_compact_gt_count(in, threshold, n, part_words, count, chunk, ws, s)
                       : launch_compact_count<kCountThreads, kCountStageParts, kCountStages>(flags, n, part_words,
                                                                                           count, chunk, ws, s);
    if (e != cudaSuccess) return e;
    const uint32_t *mask = part_words, *off = part_words + static_cast<size_t>(parts) * 17;
    const uint32_t *carry = ws.tile_sums + kMaxCountBlocks;
    const unsigned wblocks = (parts + kWriteWarps * kWritePartsPerWarp - 1) / (kWriteWarps * kWritePartsPerWarp);
    const ChunkDiv cd = chunk_div(chunk, parts);
    return out_aligned ? launch_dependent(compact_write_kernel<true, kWriteMinBlocks>, wblocks, kWriteWarps * 32, s, in,
                                          out, n, parts, cd, mask, off, carry)
                       : launch_dependent(compact_write_kernel<false, kWriteMinBlocks>, wblocks, kWriteWarps * 32, s,
                                          in, out, n, parts, cd, mask, off, carry);
}

// Ring depths measured on GB300 at 2^26: flags pass A (8 KB per tile) with
// 3 A and 3 B buffers; the fused predicate (32 KB per tile in both passes)
// with 2 A and 3 B buffers (100 against 114 us at 99% kept than 3 and 2).
using CompactPipe = CompactPolicy<16, 4, 4, 3, 3, 8, 1>;
using CompactGtPipe = CompactGtPolicy<16, 4, 4, 2, 3, 10, 1>;
constexpr unsigned kCompactWaitLimit = 1u << 18;
constexpr size_t kCompactPipelineMinN = size_t(1) << 19;   // (the two-launch path takes over from kCompactTwoPassMinN)

cudaError_t launch_compact(const int32_t *in, const uint8_t *flags, int32_t *out, int32_t *count, size_t n,
                           int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s, uint32_t *part_words)
{
    const bool out_aligned = reinterpret_cast<uintptr_t>(out) % 16 == 0;
    const uint32_t *vin = reinterpret_cast<const uint32_t *>(in);
    uint32_t *vout = reinterpret_cast<uint32_t *>(out);
    const bool bulk_ok = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(flags) % 16 == 0);
    if (bulk_ok && part_words != nullptr &&
        (carry == kCarryL2Resident || (carry == kCarryDefault && n >= kCompactTwoPassMinN)))
        return launch_compact_two_pass(vin, flags, vout, count, n, out_aligned, part_words, ws, s);
    const bool pipelined =
        bulk_ok && (carry == kCarryPipelined || (carry != kCarryLookback && n >= kCompactPipelineMinN));
    if (pipelined) {
        using G = PipeShape<CompactPipe>;
        auto kernel = pipeline_l2_kernel<CompactPipe>;
        static std::atomic<unsigned long long> attribute_set{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const unsigned long long bit = 1ull << (dev & 63);
        if ((attribute_set.load() & bit) == 0) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(G::kSmemBytes));
            if (e != cudaSuccess) return e;
            attribute_set.fetch_or(bit);
        }
        const unsigned tiles = tiles_for(n, CompactPipe::kTile);
        const unsigned grid = tiles < static_cast<unsigned>(ws.num_sms) ? tiles : static_cast<unsigned>(ws.num_sms);
        CompactPipe::Args args{vin, flags, vout, count, n, tiles, out_aligned};
        kernel<<<grid, G::kThreads, G::kSmemBytes, s>>>(args, tiles, ws.status, ws.state, ws.capacity, spin_limit,
                                                        kCompactWaitLimit);
        return cudaGetLastError();
    }
    constexpr int THREADS = kCompactThreads, VECS = kCompactVecs;
    const unsigned tiles = tiles_for(n, kCompactTile);
    const bool aligned = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(flags) % 4 == 0);
    if (aligned && out_aligned)
        compact_kernel<THREADS, VECS, true, true><<<tiles, THREADS, 0, s>>>(
            vin, flags, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    else if (aligned)
        compact_kernel<THREADS, VECS, true, false><<<tiles, THREADS, 0, s>>>(
            vin, flags, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    else if (out_aligned)
        compact_kernel<THREADS, VECS, false, true><<<tiles, THREADS, 0, s>>>(
            vin, flags, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    else
        compact_kernel<THREADS, VECS, false, false><<<tiles, THREADS, 0, s>>>(
            vin, flags, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    return cudaGetLastError();
}

template <class P>
cudaError_t set_pipeline_smem(void (*kernel)(typename P::Args, unsigned, unsigned long long *, DevState *, unsigned,
                                             unsigned, unsigned),
                              std::atomic<unsigned long long> &attribute_set)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if ((attribute_set.load() & bit) == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(PipeShape<P>::kSmemBytes));
        if (e != cudaSuccess) return e;
        attribute_set.fetch_or(bit);
    }
    return cudaSuccess;
}

cudaError_t launch_compact_gt(const int32_t *in, int32_t threshold, int32_t *out, int32_t *count, size_t n,
                              int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s,
                              uint32_t *part_words)
{
    const bool out_aligned = reinterpret_cast<uintptr_t>(out) % 16 == 0;
    const bool in_aligned = reinterpret_cast<uintptr_t>(in) % 16 == 0;
    const uint32_t *vin = reinterpret_cast<const uint32_t *>(in);
    uint32_t *vout = reinterpret_cast<uint32_t *>(out);
    if (in_aligned && part_words != nullptr && carry == kCarryL2Resident)
        return launch_compact_two_pass(vin, nullptr, vout, count, n, out_aligned, part_words, ws, s, true, threshold);
    const bool pipelined =
        in_aligned && (carry == kCarryPipelined || (carry != kCarryLookback && n >= kCompactPipelineMinN));
    if (pipelined) {
        using G = PipeShape<CompactGtPipe>;
        auto kernel = pipeline_l2_kernel<CompactGtPipe>;
        static std::atomic<unsigned long long> attribute_set{0};
        cudaError_t e = set_pipeline_smem<CompactGtPipe>(kernel, attribute_set);
        if (e != cudaSuccess) return e;
        const unsigned tiles = tiles_for(n, CompactGtPipe::kTile);
        const unsigned grid = tiles < static_cast<unsigned>(ws.num_sms) ? tiles : static_cast<unsigned>(ws.num_sms);
        CompactGtPipe::Args args{vin, threshold, vout, count, n, tiles, out_aligned};
        if (carry != kCarryDefault) {   // the pipeline alone
            kernel<<<grid, G::kThreads, G::kSmemBytes, s>>>(args, tiles, ws.status, ws.state, ws.capacity,
                                                            spin_limit, kCompactWaitLimit);
            return cudaGetLastError();
        }
        // by default the kernel first tries the one-pass capture, which needs
        // every block resident for its grid barrier: a cooperative launch
        args.capture_chunk = capture_chunk(n, grid, G::kThreads / 32);
        args.block_sums = ws.tile_sums;
        unsigned long long *status = ws.status;
        DevState *state = ws.state;
        unsigned capacity = ws.capacity, wait_limit = kCompactWaitLimit;
        void *kargs[] = {&args, const_cast<unsigned *>(&tiles), &status, &state, &capacity, &spin_limit, &wait_limit};
        return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kernel), dim3(grid), dim3(G::kThreads), kargs,
                                           G::kSmemBytes, s);
    }
    constexpr int THREADS = kCompactThreads, VECS = kCompactVecs;
    const unsigned tiles = tiles_for(n, kCompactTile);
    if (in_aligned && out_aligned)
        compact_kernel<THREADS, VECS, true, true, true><<<tiles, THREADS, 0, s>>>(
            vin, nullptr, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, threshold);
    else if (in_aligned)
        compact_kernel<THREADS, VECS, true, false, true><<<tiles, THREADS, 0, s>>>(
            vin, nullptr, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, threshold);
    else if (out_aligned)
        compact_kernel<THREADS, VECS, false, true, true><<<tiles, THREADS, 0, s>>>(
            vin, nullptr, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, threshold);
    else
        compact_kernel<THREADS, VECS, false, false, true><<<tiles, THREADS, 0, s>>>(
            vin, nullptr, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, threshold);
    return cudaGetLastError();
}

}  // namespace devscan
