// One-bit split policy of the persistent two-pass pipeline (sm_103a), and the
// zero-count helper both split kernels use.
#pragma once

#include <type_traits>

#include "core.cuh"
#include "pipeline_l2.cuh"
#include "stage.cuh"

namespace devscan {

__device__ __forceinline__ unsigned zeros_of(uint4 q, int bit)
{
    return 4u - (((q.x >> bit) & 1u) + ((q.y >> bit) & 1u) + ((q.z >> bit) & 1u) + ((q.w >> bit) & 1u));
}

// ---------------------------------------------------------------------------
// Pipelined split (see pipeline_l2.cuh): pass A reads the tile's keys and
// counts, for each consume warp's 512-key part, the keys whose bit is 0 (the
// tile's sum is the aggregate the look-back carries) and, inside a sort, the
// zeros of the next bit.  Pass B re-reads the keys (from L2); every consume
// warp, on its own, ranks its part, stages its zeros and its ones in a
// private shared-memory area and writes two contiguous runs: zeros at the
// tile's prefix plus the zeros of the earlier parts, ones at
// Z + (keys before the part - zeros before the part).  HBM traffic: 8 bytes
// per key.
// ---------------------------------------------------------------------------

// One consume warp's part of a split (bit j of zmask[q] marks key x[q][j] as
// a zero; part_len keys are real; 128 * VECS keys in a whole part): ranks the
// zeros with one scan of the rows' counts packed four to a word (a byte per
// row: a row holds at most 128 keys), stages the zeros from word zeros_at % 4
// and the ones from the next 16-byte boundary after them (plus ones_at % 4)
// in its private `stage` area (128 * VECS + 12 words), and writes both runs
// out in whole 128-bit chunks where they line up.
// COUNT_NEXT: the writes also count the keys whose bit next_bit is 0 by the
// (128 * VECS)-position output part they land in, and add those counts to
// next_cnt[part] (at most four atomics per part).
template <int VECS, bool COUNT_NEXT = false>
__device__ __forceinline__ void split_write_warp(const uint32_t (&x)[VECS][4], const uint32_t (&zmask)[VECS],
                                                 unsigned part_len, size_t zeros_at, size_t ones_at, int lane,
                                                 uint32_t *stage, uint32_t *out, bool out_aligned, size_t n,
                                                 int next_bit = 0, uint32_t *next_cnt = nullptr)
{
    static_assert(VECS == 4 || VECS == 8, "whole words of four row counts");
    constexpr int WORDS = VECS / 4;
    constexpr int PART = 128 * VECS;
    constexpr int kPartShift = VECS == 4 ? 9 : 10;
    uint32_t packed[WORDS], inc[WORDS], excl[WORDS], tot[WORDS];
#pragma unroll
    for (int w = 0; w < WORDS; ++w) {
        packed[w] = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) packed[w] |= static_cast<uint32_t>(__popc(zmask[4 * w + q])) << (8 * q);
        inc[w] = packed[w];
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
        for (int w = 0; w < WORDS; ++w) {
            const uint32_t u = __shfl_up_sync(kFullMask, inc[w], d);
            if (lane >= d) inc[w] += u;
        }
    }
    uint32_t zeros = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) {
        excl[w] = inc[w] - packed[w];
        tot[w] = __shfl_sync(kFullMask, inc[w], 31);
        zeros += (tot[w] & 0xffu) + ((tot[w] >> 8) & 0xffu) + ((tot[w] >> 16) & 0xffu) + (tot[w] >> 24);
    }
    const unsigned z_phase = out_aligned ? static_cast<unsigned>(zeros_at & 3) : 0u;
    const unsigned o_phase = out_aligned ? static_cast<unsigned>(ones_at & 3) : 0u;
    const unsigned o_base = out_aligned ? ((z_phase + zeros + 3u) & ~3u) : zeros;
    // one store per key, its slot chosen by a select (a branch per key
    // diverges on random bits); whole parts (all but the input's last) take
    // a copy of the loop without the bounds test
    const uint32_t o0 = o_base + o_phase;
    auto stage_keys = [&](auto whole_part) {
        constexpr bool WHOLE = decltype(whole_part)::value;
        uint32_t row_base = 0;
#pragma unroll
        for (int q = 0; q < VECS; ++q) {
            uint32_t zr = row_base + ((excl[q / 4] >> (8 * (q % 4))) & 0xffu);
            const uint32_t li0 = static_cast<uint32_t>((q * 32 + lane) * 4);   // index inside the part
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t li = li0 + j;
                const uint32_t z = (zmask[q] >> j) & 1u;
                const uint32_t pos = z ? z_phase + zr : o0 + (li - zr);
                if (WHOLE || li < part_len) stage[pos] = x[q][j];
                zr += z;
            }
            row_base += (tot[q / 4] >> (8 * (q % 4))) & 0xffu;
        }
    };
    if (part_len == static_cast<unsigned>(PART))
        stage_keys(std::true_type{});
    else
        stage_keys(std::false_type{});
    __syncwarp();
    if (COUNT_NEXT) {
        // also count bit next_bit's zeros by the output part they land in
        uint32_t c[4] = {0u, 0u, 0u, 0u};
        if (out_aligned) {
            write_run_direct_count<32, PART>(out, zeros_at, zeros, stage, lane, n, next_bit, c[0], c[1]);
            write_run_direct_count<32, PART>(out, ones_at, part_len - zeros, stage + o_base, lane, n, next_bit, c[2],
                                             c[3]);
        } else {
            write_run_scalar_count<32, PART>(out, zeros_at, zeros, stage, 0, lane, n, next_bit, c[0], c[1]);
            write_run_scalar_count<32, PART>(out, ones_at, part_len - zeros, stage, static_cast<int>(zeros), lane, n,
                                             next_bit, c[2], c[3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = __reduce_add_sync(kFullMask, c[i]);
        if (lane == 0) {
            const size_t zp = zeros_at >> kPartShift, op = ones_at >> kPartShift;
            if (c[0] != 0) atomicAdd(next_cnt + zp, c[0]);
            if (c[1] != 0) atomicAdd(next_cnt + zp + 1, c[1]);
            if (c[2] != 0) atomicAdd(next_cnt + op, c[2]);
            if (c[3] != 0) atomicAdd(next_cnt + op + 1, c[3]);
        }
    } else if (out_aligned) {
        write_run_direct<32>(out, zeros_at, zeros, stage, lane, n);
        write_run_direct<32>(out, ones_at, part_len - zeros, stage + o_base, lane, n);
    } else {
        write_run_scalar<32>(out, zeros_at, zeros, stage, 0, lane, n);
        write_run_scalar<32>(out, ones_at, part_len - zeros, stage, static_cast<int>(zeros), lane, n);
    }
    __syncwarp();   // the area is read before the warp stages its next part
}

template <int NS_, int NR_, int VECS_, int SA_, int SB_, int R_, int PREFETCH = 0>
struct SplitPolicy {
    using Op = AddU32;
    using S = uint32_t;
    static constexpr int kAHint = kL2EvictLast, kBHint = kL2EvictFirst, kPrefetch = PREFETCH;
    static constexpr int kConsumeWarps = NS_, kReduceWarps = NR_, kRecords = R_, kAStages = SA_, kBStages = SB_;
    static constexpr int VECS = VECS_;
    static constexpr int kWarpItems = 32 * 4 * VECS;
    static constexpr int kTile = NS_ * 32 * 4 * VECS;
    static constexpr size_t kABytes = static_cast<size_t>(kTile) * 4;
    static constexpr size_t kBBytes = static_cast<size_t>(kTile) * 4;
    static constexpr int kParts = NS_;                   // one part per consume warp
    static constexpr bool kWarpIndependent = true;       // no barrier in consume()
    // words: the zeros from word 0..3, the ones from the next 16-byte boundary
    // plus 0..3, and the copy-out's last whole chunk: at most kWarpItems + 12
    static constexpr int kWarpStage = kWarpItems + 12;
    static constexpr size_t kScratchBytes = static_cast<size_t>(NS_) * kWarpStage * 4;
    static constexpr bool kHasExtra = true;
    struct Args {
        const uint32_t *keys;
        uint32_t *out;
        size_t n;
        int bit;
        const unsigned *zeros_total;
        unsigned *next_zeros;   // may be null
        int next_bit;
        bool out_aligned;
    };
    __device__ static unsigned tile_len(const Args &a, unsigned t)
    {
        const size_t rem = a.n - static_cast<size_t>(t) * kTile;
        return rem < static_cast<size_t>(kTile) ? static_cast<unsigned>(rem) : static_cast<unsigned>(kTile);
    }
    __device__ static unsigned copied(const Args &a, unsigned t) { return tile_len(a, t) & ~3u; }
    __device__ static const void *a_src(const Args &a, unsigned t) { return a.keys + static_cast<size_t>(t) * kTile; }
    __device__ static unsigned a_bytes(const Args &a, unsigned t) { return copied(a, t) * 4u; }
    __device__ static void prefetch_l2(const Args &a, unsigned t, uint64_t pol)
    {
        if (a_bytes(a, t) != 0) bulk_prefetch_l2(a_src(a, t), a_bytes(a, t), pol);
    }
    __device__ static void b_copies(const Args &a, unsigned t, const void **src, unsigned *bytes, unsigned *off)
    {
        src[0] = a.keys + static_cast<size_t>(t) * kTile;
        bytes[0] = copied(a, t) * 4u;
        off[0] = 0;
    }
    __device__ static void reduce_parts(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int, S &v,
                                        unsigned &extra, uint32_t *part)
    {
        static_assert(NS_ % NR_ == 0 && kWarpItems / 4 % 32 == 0, "whole parts per reduce warp");
        constexpr int PPW = NS_ / NR_, CH = kWarpItems / 4 / 32;   // parts per warp, 4-key chunks per lane
        const int lane = rtid & 31, rw = rtid >> 5;
        const unsigned cp = copied(a, t), len = tile_len(a, t);
        const size_t base = static_cast<size_t>(t) * kTile;
        const uint4 *k4 = reinterpret_cast<const uint4 *>(abuf);
        const uint32_t *k1 = reinterpret_cast<const uint32_t *>(abuf);
        unsigned c[PPW], nz = 0;
        if (len == static_cast<unsigned>(kTile)) {
            const bool next = a.next_zeros != nullptr;   // the next bit's zeros are wanted (inside a sort)
            if (next && a.next_bit == a.bit + 1) {
                // both bits from one shift: bit b counts 1 and bit b+1 counts
                // 32 in one accumulator (at most 16 keys per lane and part)
#pragma unroll
                for (int i = 0; i < PPW; ++i) {
                    uint32_t ones = 0;
#pragma unroll
                    for (int k = 0; k < CH; ++k) {
                        const uint4 q = k4[(rw + i * NR_) * (kWarpItems / 4) + k * 32 + lane];
                        const uint32_t t0 = (q.x >> a.bit) & 3u, t1 = (q.y >> a.bit) & 3u;
                        const uint32_t t2 = (q.z >> a.bit) & 3u, t3 = (q.w >> a.bit) & 3u;
                        ones += (t0 + (t0 & 2u) * 15u) + (t1 + (t1 & 2u) * 15u) + (t2 + (t2 & 2u) * 15u) +
                                (t3 + (t3 & 2u) * 15u);
                    }
                    c[i] = 4u * CH - (ones & 31u);
                    nz += 4u * CH - (ones >> 5);
                }
            } else {
#pragma unroll
                for (int i = 0; i < PPW; ++i) {
                    c[i] = 0;
#pragma unroll
                    for (int k = 0; k < CH; ++k) {
                        const uint4 q = k4[(rw + i * NR_) * (kWarpItems / 4) + k * 32 + lane];
                        c[i] += zeros_of(q, a.bit);
                        if (next) nz += zeros_of(q, a.next_bit);
                    }
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < PPW; ++i) {
                c[i] = 0;
                for (int k = 0; k < CH; ++k) {
                    const unsigned e = static_cast<unsigned>((rw + i * NR_) * kWarpItems + 4 * (k * 32 + lane));
                    for (unsigned j = 0; j < 4; ++j)
                        if (e + j < len) {
                            const uint32_t key = (e + j < cp) ? k1[e + j] : a.keys[base + e + j];
                            c[i] += ((key >> a.bit) & 1u) ? 0u : 1u;
                            nz += ((key >> a.next_bit) & 1u) ? 0u : 1u;
                        }
                }
            }
        }
        const unsigned mine = store_part_counts<PPW, NR_>(c, rw, lane, part);
        v = (lane == 0) ? mine : 0u;
        extra = nz;
    }
    __device__ static void after_reduce(const Args &a, unsigned, unsigned next_zero_count)
    {
        if (a.next_zeros != nullptr && next_zero_count != 0) atomicAdd(a.next_zeros, next_zero_count);
    }
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *, uint32_t *, int warp,
                                       int lane, Release &release)
    {
        const unsigned t = ct.tile;
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        const uint32_t *buf = reinterpret_cast<const uint32_t *>(ct.buf);
        const unsigned len = tile_len(a, t), cp = copied(a, t);
        uint32_t x[VECS][4], zmask[VECS];
#pragma unroll
        for (int q = 0; q < VECS; ++q) {
            if (len == static_cast<unsigned>(kTile)) {
                const uint4 u = reinterpret_cast<const uint4 *>(buf + wbase)[q * 32 + lane];
                x[q][0] = u.x;
                x[q][1] = u.y;
                x[q][2] = u.z;
                x[q][3] = u.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const unsigned e = static_cast<unsigned>(wbase + (q * 32 + lane) * 4 + j);
                    x[q][j] = (e < cp) ? buf[e] : ((e < len) ? a.keys[base + e] : 0u);
                }
            }
            uint32_t m = 0;
            if (len == static_cast<unsigned>(kTile)) {
                // bit j: key j's bit is 0 (the ones' bits gathered, then flipped)
#pragma unroll
                for (int j = 0; j < 4; ++j) m |= ((x[q][j] >> a.bit) & 1u) << j;
                m ^= 0xfu;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const unsigned e = static_cast<unsigned>(wbase + (q * 32 + lane) * 4 + j);
                    if (e < len && !((x[q][j] >> a.bit) & 1u)) m |= 1u << j;
                }
            }
            zmask[q] = m;
        }
        // the zero total is fixed for the launch: one global read per warp,
        // kept (plus one, so that 0 means "not read yet") in the warp's word
        if (*ct.warp_state == 0) *ct.warp_state = *a.zeros_total + 1u;
        const size_t zeros_at = static_cast<size_t>(ct.prefix) + ct.part_excl[warp];
        const size_t ones_at = static_cast<size_t>(*ct.warp_state - 1u) + (base + wbase - zeros_at);
        const unsigned part_len = len > static_cast<unsigned>(wbase)
                                      ? (len - wbase < static_cast<unsigned>(kWarpItems) ? len - wbase
                                                                                          : static_cast<unsigned>(kWarpItems))
                                      : 0u;
        release();   // keys in registers, offsets read: the B buffer and the record are free
        uint32_t *stage = reinterpret_cast<uint32_t *>(ct.scratch) + warp * kWarpStage;
        split_write_warp<VECS>(x, zmask, part_len, zeros_at, ones_at, lane, stage, a.out, a.out_aligned, a.n);
        return 0;   // no warp-totals buffer used
    }
};

}  // namespace devscan
