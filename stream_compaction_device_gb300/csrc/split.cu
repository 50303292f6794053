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
// anyway): a block per SM streams its chunk of 1,024-key parts through shared
// memory, counts every part's zeros and turns the counts into offsets within
// the chunk; the last block to finish scans the chunk totals into chunk
// carries and the total Z.  The write launch, a programmatic dependent of the
// count (its keys load while the count ends), gives a warp per part: it ranks
// its keys and writes its zeros run at its offset plus its chunk's carry and
// its ones run at Z + (keys before the part - that offset).  The same bytes as
// the count pass plus the pipelined split (12 per key), without a chain
// between tiles.
// ---------------------------------------------------------------------------
constexpr int kSplitPart = 1024, kSplitCountThreads = 512, kSplitStageParts = 16, kSplitStages = 3,
              kSplitWriteWarps = 8;
constexpr int kSplitRows = kSplitPart / 128;   // 16-byte loads per lane and part
constexpr unsigned kSplitCountWaitLimit = 1u << 18;
constexpr unsigned kSplitMaxCountBlocks = 512;   // chunk totals and carries share the workspace's tile sums
constexpr int kSortOffsetThreads = 1024;

// off[p]: zeros of bit `bit` in the parts before p in its chunk.  Block b
// takes the chunk of parts [b * chunk, (b + 1) * chunk): its whole parts
// stream through NSTG shared-memory stages of SP parts (dynamic shared
// memory), the ragged last part of the input takes plain loads.  The last
// block writes carry[b] = zeros in the chunks before b, and *zeros = all
// zeros (block_sums: one word per block).
template <int THREADS, int SP, int NSTG>
__global__ void __launch_bounds__(THREADS, 1)
split_count_kernel(const uint32_t *__restrict__ keys, size_t n, int bit, unsigned parts, unsigned chunk,
                   uint32_t *__restrict__ off, uint32_t *__restrict__ block_sums, uint32_t *__restrict__ carry,
                   unsigned *__restrict__ zeros, DevState *st)
{
    static_assert(THREADS >= static_cast<int>(kSplitMaxCountBlocks), "the last block scans one chunk total per thread");
    constexpr int NW = THREADS / 32;
    extern __shared__ __align__(128) uint8_t s_ring[];
    __shared__ uint64_t s_full[NSTG];
    __shared__ uint32_t s_w[NW];
    allow_dependent_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned p0 = blockIdx.x * chunk, p1 = p0 + chunk < parts ? p0 + chunk : parts;
    const unsigned whole = static_cast<unsigned>(n / kSplitPart);
    const unsigned q1 = p1 < whole ? p1 : (p0 > whole ? p0 : whole);   // [p0, q1): whole parts
    // phase 1: a part per warp; lane L reads the part's 16-byte groups L, L + 32, L + 64, ...
    const bool streamed = stream_parts<kSplitPart * 4, SP, NSTG>(
        reinterpret_cast<const uint8_t *>(keys), p0, q1, s_ring, s_full, kSplitCountWaitLimit,
        [&](unsigned p, const uint8_t *part) {
            const uint4 *k4 = reinterpret_cast<const uint4 *>(part);
            uint32_t z = 0;
#pragma unroll
            for (int g = 0; g < kSplitRows; ++g) z += zeros_of(k4[g * 32 + lane], bit);
            z = __reduce_add_sync(kFullMask, z);
            if (lane == 0) off[p] = z;
        });
    if (!streamed && tid == 0) atomicOr(&st->error, kErrTimeout);
    for (unsigned p = q1 + warp; p < p1; p += NW) {   // the input's ragged last part
        const size_t e0 = static_cast<size_t>(p) * kSplitPart;
        uint32_t z = 0;
        for (size_t e = e0 + lane; e < n && e < e0 + kSplitPart; e += 32) z += ((keys[e] >> bit) & 1u) ? 0u : 1u;
        z = __reduce_add_sync(kFullMask, z);
        if (lane == 0) off[p] = z;
    }
    __syncthreads();   // every part's count written

    // phase 2: the counts become offsets within the chunk, in place, THREADS parts at a time
    uint32_t run = 0;
    for (unsigned base = p0; base < p1; base += THREADS) {
        const unsigned p = base + tid;
        const uint32_t c = p < p1 ? off[p] : 0u;   // this thread's own part: read before it is overwritten
        uint32_t total;
        const uint32_t excl = block_excl_scan<THREADS>(c, s_w, tid, total);
        if (p < p1) off[p] = run + excl;
        run += total;
        __syncthreads();   // s_w is read before the next round writes it
    }
    uint32_t all;
    if (last_block_carries<THREADS>(run, block_sums, carry, st, s_w, all) && tid == 0) *zeros = all;
}

// Warp w of block b splits part b * kSplitWriteWarps + w.  COUNT_NEXT: it
// also adds, per part of `out`, the keys it writes there whose bit next_bit
// is 0 to next_cnt (the next pass's part counts, in a sort).  Four blocks per
// SM (64 registers).
template <bool OUT_ALIGNED, bool COUNT_NEXT>
__global__ void __launch_bounds__(kSplitWriteWarps * 32, 4)
split_write_kernel(const uint32_t *__restrict__ keys, uint32_t *__restrict__ out, size_t n, int bit, unsigned parts,
                   ChunkDiv chunk, const uint32_t *off, const uint32_t *carry, const unsigned *zeros,
                   int next_bit, uint32_t *__restrict__ next_cnt)
{
    constexpr int kStage = kSplitPart + 12;   // the zeros, the ones from the next 16-byte boundary, a spare chunk
    __shared__ __align__(16) uint32_t s_stage[kSplitWriteWarps][kStage];
    // a sort's next offsets launch may start once every block has begun: it
    // waits for this grid to finish before it reads the counts
    allow_dependent_launch();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned p = blockIdx.x * kSplitWriteWarps + warp;
    if (p >= parts) return;   // the whole warp: no barrier follows
    const size_t b = static_cast<size_t>(p) * kSplitPart;
    const unsigned part_len = n - b < static_cast<size_t>(kSplitPart) ? static_cast<unsigned>(n - b) : kSplitPart;
    uint32_t x[kSplitRows][4], zmask[kSplitRows];
    if (part_len == static_cast<unsigned>(kSplitPart)) {
        const uint4 *k4 = reinterpret_cast<const uint4 *>(keys + b);
        const uint32_t sel = byte_sel(bit);
#pragma unroll
        for (int q = 0; q < kSplitRows; ++q) {
            const uint4 u = __ldcs(k4 + q * 32 + lane);
            x[q][0] = u.x;
            x[q][1] = u.y;
            x[q][2] = u.z;
            x[q][3] = u.w;
            zmask[q] = nibble_at_bit(u, sel, bit & 7) ^ 0xfu;
        }
    } else {
#pragma unroll
        for (int q = 0; q < kSplitRows; ++q) {
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
    wait_primary_grid();   // the count launch's offsets, carries and Z (the keys need no wait)
    const size_t zeros_at = static_cast<size_t>(off[p]) + carry[chunk.of(p)];
    const size_t ones_at = static_cast<size_t>(*zeros) + (b - zeros_at);
    split_write_warp<kSplitRows, COUNT_NEXT>(x, zmask, part_len, zeros_at, ones_at, lane, s_stage[warp], out, OUT_ALIGNED, n,
                                    next_bit, next_cnt);
}

// A sort pass's offsets from the part counts the previous pass's writes
// gathered: off[p] = counts of the parts before p in its chunk (block b takes
// parts [b * chunk, (b + 1) * chunk)); the last block writes carry[b] and
// *zeros = all counts.  Each count is reset to 0 once read, ready for the
// next pass's writes.
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
part_offsets_kernel(uint32_t *cnt, unsigned parts, unsigned chunk, uint32_t *__restrict__ off,
                    uint32_t *__restrict__ block_sums, uint32_t *__restrict__ carry, unsigned *__restrict__ zeros,
                    DevState *st)
{
    static_assert(THREADS >= static_cast<int>(kSplitMaxCountBlocks), "the last block scans one chunk total per thread");
    __shared__ uint32_t s_w[THREADS / 32];
    // launched as a programmatic dependent of the previous pass's write
    // launch: wait for its counts (and its keys) to be complete before this
    // grid lets the next write launch start, as that one reads those keys
    // before its own wait
    wait_primary_grid();
    allow_dependent_launch();
    const int tid = threadIdx.x;
    const unsigned p0 = blockIdx.x * chunk, p1 = p0 + chunk < parts ? p0 + chunk : parts;
    uint32_t run = 0;
    for (unsigned base = p0; base < p1; base += THREADS) {
        const unsigned p = base + tid;
        uint32_t c = 0;
        if (p < p1) {
            c = cnt[p];
            cnt[p] = 0;
        }
        uint32_t total;
        const uint32_t excl = block_excl_scan<THREADS>(c, s_w, tid, total);
        if (p < p1) off[p] = run + excl;
        run += total;
        __syncthreads();   // s_w is read before the next round writes it
    }
    uint32_t all;
    if (last_block_carries<THREADS>(run, block_sums, carry, st, s_w, all) && tid == 0) *zeros = all;
}

size_t split_part_words(size_t n) { return (n + kSplitPart - 1) / kSplitPart; }

// The count launch: THREADS per block, NSTG * SP * 2048 bytes of stages;
// `chunk` parts per block.  The workspace's tile sums hold the chunk totals
// (first kSplitMaxCountBlocks words) and carries (next).
template <int THREADS, int SP, int NSTG>
cudaError_t launch_split_count(const uint32_t *keys, size_t n, int bit, uint32_t *off, unsigned *zeros, unsigned chunk,
                               const Workspace &ws, cudaStream_t s)
{
    static std::atomic<unsigned long long> smem_set{0};
    constexpr int kSmem = NSTG * SP * kSplitPart * 4;
    auto kernel = split_count_kernel<THREADS, SP, NSTG>;
    cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void *>(kernel), kSmem, smem_set);
    if (e != cudaSuccess) return e;
    const unsigned parts = static_cast<unsigned>(split_part_words(n));
    const unsigned blocks = (parts + chunk - 1) / chunk;
    kernel<<<blocks, THREADS, kSmem, s>>>(keys, n, bit, parts, chunk, off, ws.tile_sums,
                                          ws.tile_sums + kSplitMaxCountBlocks, zeros, ws.state);
    return cudaGetLastError();
}

// Parts per chunk: one chunk per SM (fewer for small inputs, at least a part
// per warp each), at most kSplitMaxCountBlocks chunks.
unsigned split_count_chunk(unsigned parts, unsigned warps, int num_sms)
{
    unsigned blocks = std::min<unsigned>(static_cast<unsigned>(num_sms), kSplitMaxCountBlocks);
    blocks = std::min(blocks, (parts + warps - 1) / warps);
    return (parts + blocks - 1) / blocks;
}

// The write launch, a programmatic dependent of the launch that produced
// off, carry and *zeros; next_cnt non-null: also count bit next_bit's zeros
// per part of `out`.
cudaError_t launch_split_write(const uint32_t *keys, uint32_t *out, size_t n, int bit, unsigned chunk,
                               const uint32_t *off, const uint32_t *carry, const unsigned *zeros, int next_bit,
                               uint32_t *next_cnt, cudaStream_t s)
{
    const unsigned parts = static_cast<unsigned>(split_part_words(n));
    const unsigned wblocks = (parts + kSplitWriteWarps - 1) / kSplitWriteWarps;
    const bool aligned = reinterpret_cast<uintptr_t>(out) % 16 == 0;
    const ChunkDiv cd = chunk_div(chunk, parts);
    constexpr unsigned kThreads = kSplitWriteWarps * 32;
    if (next_cnt != nullptr)
        return aligned ? launch_dependent(split_write_kernel<true, true>, wblocks, kThreads, s, keys, out, n, bit, parts,
                                          cd, off, carry, zeros, next_bit, next_cnt)
                       : launch_dependent(split_write_kernel<false, true>, wblocks, kThreads, s, keys, out, n, bit,
                                          parts, cd, off, carry, zeros, next_bit, next_cnt);
    return aligned ? launch_dependent(split_write_kernel<true, false>, wblocks, kThreads, s, keys, out, n, bit, parts,
                                      cd, off, carry, zeros, 0, static_cast<uint32_t *>(nullptr))
                   : launch_dependent(split_write_kernel<false, false>, wblocks, kThreads, s, keys, out, n, bit, parts,
                                      cd, off, carry, zeros, 0, static_cast<uint32_t *>(nullptr));
}

cudaError_t launch_split_two_pass(const uint32_t *keys, uint32_t *out, size_t n, int bit, unsigned *zeros,
                                  uint32_t *part_words, const Workspace &ws, cudaStream_t s)
{
    const unsigned parts = static_cast<unsigned>(split_part_words(n));
    const unsigned chunk = split_count_chunk(parts, kSplitCountThreads / 32, ws.num_sms);
    cudaError_t e = launch_split_count<kSplitCountThreads, kSplitStageParts, kSplitStages>(keys, n, bit, part_words,
                                                                                          zeros, chunk, ws, s);
    if (e != cudaSuccess) return e;
    return launch_split_write(keys, out, n, bit, chunk, part_words, ws.tile_sums + kSplitMaxCountBlocks, zeros, 0,
                              nullptr, s);
}

size_t sort_part_words(size_t n) { return 2 * split_part_words(n); }

cudaError_t launch_sort_two_pass(uint32_t *keys, uint32_t *tmp, size_t n, unsigned *zeros, uint32_t *part_words,
                                 const Workspace &ws, cudaStream_t s)
{
    const unsigned parts = static_cast<unsigned>(split_part_words(n));
    const unsigned chunk = split_count_chunk(parts, kSplitCountThreads / 32, ws.num_sms);
    uint32_t *off = part_words, *cnt = part_words + parts;
    const uint32_t *carry = ws.tile_sums + kSplitMaxCountBlocks;
    cudaError_t e = cudaMemsetAsync(cnt, 0, static_cast<size_t>(parts) * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    e = launch_split_count<kSplitCountThreads, kSplitStageParts, kSplitStages>(keys, n, 0, off, zeros, chunk, ws, s);
    if (e != cudaSuccess) return e;
    const uint32_t *src = keys;
    uint32_t *dst = tmp;
    for (int bit = 0; bit < 32; ++bit) {
        e = launch_split_write(src, dst, n, bit, chunk, off, carry, zeros, bit + 1, bit < 31 ? cnt : nullptr, s);
        if (e != cudaSuccess) return e;
        if (bit < 31) {
            const unsigned blocks = (parts + chunk - 1) / chunk;
            e = launch_dependent(part_offsets_kernel<kSortOffsetThreads>, blocks, kSortOffsetThreads, s, cnt, parts,
                                 chunk, off, ws.tile_sums, ws.tile_sums + kSplitMaxCountBlocks, zeros, ws.state);
            if (e != cudaSuccess) return e;
        }
        src = dst;
        dst = (dst == tmp) ? keys : tmp;
    }
    return cudaSuccess;
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
