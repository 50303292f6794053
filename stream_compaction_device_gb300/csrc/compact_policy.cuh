// Compaction policy of the persistent two-pass pipeline (sm_103a), and the
// byte-flag helpers both compaction kernels use.
#pragma once

#include "core.cuh"
#include "pipeline_l2.cuh"
#include "stage.cuh"
#include "capture.cuh"

namespace devscan {

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t *p) { return __ldcs(p); }

// Bit 7 of every nonzero byte of f (the other bits clear): a byte's low
// seven bits plus 0x7f reach bit 7 exactly when they are nonzero, without
// carrying into the next byte.
__device__ __forceinline__ uint32_t nonzero_byte_tops(uint32_t f)
{
    return (f | ((f & 0x7f7f7f7fu) + 0x7f7f7f7fu)) & 0x80808080u;
}

// Number of nonzero bytes of f.
__device__ __forceinline__ unsigned nonzero_bytes(uint32_t f) { return __popc(nonzero_byte_tops(f)); }

// Bit k set when byte k of f is nonzero: the four byte flags (bits 0, 8, 16,
// 24) are gathered into bits 21..24 by one multiply with 1 + 2^7 + 2^14 +
// 2^21 (no two partial products share a bit, so nothing carries).
__device__ __forceinline__ uint32_t nonzero_byte_mask(uint32_t f)
{
    return ((nonzero_byte_tops(f) >> 7) * 0x00204081u) >> 21 & 0xfu;
}

// ---------------------------------------------------------------------------
// Pipelined compaction (see pipeline_l2.cuh): pass A reads only the tile's
// flags (1 byte per element) and counts the kept elements -- the aggregate
// the look-back carries; pass B reads the values and (from L2) the flags,
// ranks the kept values, stages them in the B buffer at their tile rank and
// writes one contiguous run at the tile's prefix.  HBM traffic is the
// algorithmic 5 bytes per element plus 4 per kept element.
// ---------------------------------------------------------------------------
// Second half of a compaction consume step, shared by both predicate forms,
// run by one warp on its own part of the tile (bit j of keep[q] keeps
// x[q][j]).  The warp's kept elements form one contiguous run of the output
// starting at g0 (the tile's prefix plus the kept counts of the earlier parts,
// from pass A), so the warp needs no other warp: it ranks its elements with
// one scan of the four rows' counts packed into the bytes of a word (a row
// holds at most 128), stages them in its private `stage` area (kWarpItems + 4
// words, 16-byte aligned) in phase with their destination and copies the run
// out in whole 128-bit chunks, only the two ragged ends element by element.
template <int VECS>
__device__ __forceinline__ void compact_write_warp(const uint32_t (&x)[VECS][4], const uint32_t (&keep)[VECS],
                                                   size_t g0, int lane, uint32_t *stage, uint32_t *out,
                                                   bool out_aligned, size_t n)
{
    static_assert(VECS == 4, "the four rows' counts share one word");
    uint32_t packed = 0;
#pragma unroll
    for (int q = 0; q < VECS; ++q) packed |= static_cast<uint32_t>(__popc(keep[q])) << (8 * q);
    uint32_t inc = packed;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t u = __shfl_up_sync(kFullMask, inc, d);
        if (lane >= d) inc += u;
    }
    const uint32_t excl = inc - packed, tot = __shfl_sync(kFullMask, inc, 31);
    const unsigned phase = out_aligned ? static_cast<unsigned>(g0 & 3) : 0u;
    uint32_t row_base = phase, count = 0;
#pragma unroll
    for (int q = 0; q < VECS; ++q) {
        uint32_t rank = row_base + ((excl >> (8 * q)) & 0xffu);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if ((keep[q] >> j) & 1u) stage[rank++] = x[q][j];
        const uint32_t row_total = (tot >> (8 * q)) & 0xffu;
        row_base += row_total;
        count += row_total;
    }
    __syncwarp();
    if (out_aligned)
        write_run_direct<32>(out, g0, count, stage, lane, n);
    else
        write_run_scalar<32>(out, g0, count, stage, 0, lane, n);
    __syncwarp();   // the area is read before the warp stages its next part
}

// Pass A copies only the flags, so the values need not reach L2 before a
// tile is counted: they are moved there once pass A has counted the tile,
// while its prefix resolves.  That keeps L2's footprint smaller than moving
// them with the flags at ticket time (measured 9-10% faster at 50-99% kept;
// loading only the kept values of sparse tiles instead of the bulk copy
// measured slower).
template <int NS_, int NR_, int VECS_, int SA_, int SB_, int R_, int PREFETCH = 0>
struct CompactPolicy {
    using Op = AddU32;
    using S = uint32_t;
    static constexpr int kAHint = kL2EvictLast, kBHint = kL2EvictFirst, kPrefetch = PREFETCH;
    static constexpr int kConsumeWarps = NS_, kReduceWarps = NR_, kRecords = R_, kAStages = SA_, kBStages = SB_;
    static constexpr int VECS = VECS_;
    static constexpr int kWarpItems = 32 * 4 * VECS;
    static constexpr int kTile = NS_ * 32 * 4 * VECS;
    static constexpr size_t kValueBytes = static_cast<size_t>(kTile) * 4;
    static constexpr size_t kABytes = static_cast<size_t>(kTile);                // flags
    static constexpr size_t kBBytes = kValueBytes + static_cast<size_t>(kTile);  // values, then flags
    static constexpr bool kHasExtra = false;
    static constexpr int kParts = NS_;                                          // one part per consume warp
    static constexpr bool kWarpIndependent = true;                              // no barrier in consume()
    static constexpr bool kAggregateAware = true;                               // on_aggregate moves the values
    static constexpr int kWarpStage = kWarpItems + 4;                           // words, 16-byte multiple
    static constexpr size_t kScratchBytes = static_cast<size_t>(NS_) * kWarpStage * 4;
    struct Args {
        const uint32_t *in;
        const uint8_t *flags;
        uint32_t *out;
        int32_t *count;
        size_t n;
        unsigned num_tiles;
        bool out_aligned;
    };
    __device__ static unsigned tile_len(const Args &a, unsigned t)
    {
        const size_t rem = a.n - static_cast<size_t>(t) * kTile;
        return rem < static_cast<size_t>(kTile) ? static_cast<unsigned>(rem) : static_cast<unsigned>(kTile);
    }
    __device__ static unsigned flags_copied(const Args &a, unsigned t) { return tile_len(a, t) & ~15u; }
    __device__ static unsigned values_copied(const Args &a, unsigned t) { return tile_len(a, t) & ~3u; }
    __device__ static const void *a_src(const Args &a, unsigned t) { return a.flags + static_cast<size_t>(t) * kTile; }
    __device__ static unsigned a_bytes(const Args &a, unsigned t) { return flags_copied(a, t); }
    // the flags, for pass A (the values follow in on_aggregate)
    __device__ static void prefetch_l2(const Args &a, unsigned t, uint64_t pol)
    {
        if (flags_copied(a, t) != 0) bulk_prefetch_l2(a_src(a, t), flags_copied(a, t), pol);
    }
    // after pass A: the tile's values start moving into L2 while its prefix
    // resolves
    __device__ static void on_aggregate(const Args &a, unsigned t, uint32_t)
    {
        if (values_copied(a, t) != 0)
            bulk_prefetch_l2(a.in + static_cast<size_t>(t) * kTile, values_copied(a, t) * 4u, l2_policy_evict_last());
    }
    __device__ static void b_copies_for(const Args &a, unsigned t, uint32_t, const void **src, unsigned *bytes,
                                        unsigned *off)
    {
        b_copies(a, t, src, bytes, off);
    }
    __device__ static void b_copies(const Args &a, unsigned t, const void **src, unsigned *bytes, unsigned *off)
    {
        src[0] = a.in + static_cast<size_t>(t) * kTile;
        bytes[0] = values_copied(a, t) * 4u;
        off[0] = 0;
        src[1] = a.flags + static_cast<size_t>(t) * kTile;
        bytes[1] = flags_copied(a, t);
        off[1] = static_cast<unsigned>(kValueBytes);
    }
    // pass A: the kept count of each consume warp's part (kWarpItems flags),
    // one warp reduction per part; lane 0 of each reduce warp returns the
    // sum of its parts (the kernel adds the lanes and the warps)
    __device__ static void reduce_parts(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int,
                                        S &v, unsigned &, uint32_t *part)
    {
        static_assert(NS_ % NR_ == 0 && kWarpItems / 16 % 32 == 0, "whole parts per reduce warp");
        constexpr int PPW = NS_ / NR_, CH = kWarpItems / 16 / 32;   // parts per warp, 16-flag chunks per lane
        const int lane = rtid & 31, rw = rtid >> 5;
        const unsigned cp = flags_copied(a, t), len = tile_len(a, t);
        const size_t base = static_cast<size_t>(t) * kTile;
        const uint4 *f4 = reinterpret_cast<const uint4 *>(abuf);
        unsigned c[PPW];
        if (len == static_cast<unsigned>(kTile)) {
#pragma unroll
            for (int i = 0; i < PPW; ++i) {
                c[i] = 0;
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const uint4 q = f4[(rw + i * NR_) * (kWarpItems / 16) + k * 32 + lane];
                    c[i] += nonzero_bytes(q.x) + nonzero_bytes(q.y) + nonzero_bytes(q.z) + nonzero_bytes(q.w);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < PPW; ++i) {
                c[i] = 0;
                for (int k = 0; k < CH; ++k) {
                    const unsigned e = static_cast<unsigned>((rw + i * NR_) * kWarpItems + 16 * (k * 32 + lane));
                    for (unsigned j = 0; j < 16; ++j)
                        if (e + j < len)
                            c[i] += ((e + j < cp ? abuf[e + j] : a.flags[base + e + j]) != 0) ? 1u : 0u;
                }
            }
        }
        const unsigned mine = store_part_counts<PPW, NR_>(c, rw, lane, part);
        v = (lane == 0) ? mine : 0u;
    }
    __device__ static void after_reduce(const Args &, unsigned, unsigned) {}
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *, uint32_t *, int warp,
                                       int lane, Release &release)
    {
        const unsigned t = ct.tile;
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        const uint32_t *vals = reinterpret_cast<const uint32_t *>(ct.buf);
        const uint8_t *fl = ct.buf + kValueBytes;
        const unsigned len = tile_len(a, t);
        const unsigned vcp = values_copied(a, t), fcp = flags_copied(a, t);
        uint32_t x[VECS][4], keep[VECS];
        if (len == static_cast<unsigned>(kTile)) {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(vals + wbase);
            const uint32_t *f32 = reinterpret_cast<const uint32_t *>(fl + wbase);
#pragma unroll
            for (int q = 0; q < VECS; ++q) {
                const uint4 u = v4[q * 32 + lane];
                x[q][0] = u.x;
                x[q][1] = u.y;
                x[q][2] = u.z;
                x[q][3] = u.w;
                keep[q] = nonzero_byte_mask(f32[q * 32 + lane]);
            }
        } else {
#pragma unroll
            for (int q = 0; q < VECS; ++q) {
                uint32_t m = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const unsigned e = static_cast<unsigned>(wbase + (q * 32 + lane) * 4 + j);
                    x[q][j] = (e < vcp) ? vals[e] : ((e < len) ? a.in[base + e] : 0u);
                    const uint8_t f = (e < fcp) ? fl[e] : ((e < len) ? a.flags[base + e] : uint8_t(0));
                    if (f != 0) m |= 1u << j;
                }
                keep[q] = m;
            }
        }
        const size_t g0 = static_cast<size_t>(ct.prefix) + ct.part_excl[warp];
        release();   // values in registers, offset read: the B buffer and the record are free
        uint32_t *stage = reinterpret_cast<uint32_t *>(ct.scratch) + warp * kWarpStage;
        compact_write_warp<VECS>(x, keep, g0, lane, stage, a.out, a.out_aligned, a.n);
        if (t == a.num_tiles - 1 && warp == 0 && lane == 0) *a.count = static_cast<int32_t>(ct.prefix + ct.aggregate);
        return 0;   // no warp-totals buffer used
    }
};


// ---------------------------------------------------------------------------
// Pipelined compaction with the predicate evaluated in the kernel (keep
// in[i] when in[i] > threshold, signed): pass A reads the tile's values and
// counts the kept ones; pass B reads them again (L2 hits), re-evaluates the
// predicate, ranks, stages and writes the run.  No flag array exists, so the
// HBM traffic is 4 bytes per element plus 4 per kept element.
// ---------------------------------------------------------------------------
template <int NS_, int NR_, int VECS_, int SA_, int SB_, int R_, int PREFETCH = 0>
struct CompactGtPolicy {
    using Op = AddU32;
    using S = uint32_t;
    static constexpr int kAHint = kL2EvictLast, kBHint = kL2EvictFirst, kPrefetch = PREFETCH;
    static constexpr int kConsumeWarps = NS_, kReduceWarps = NR_, kRecords = R_, kAStages = SA_, kBStages = SB_;
    static constexpr int VECS = VECS_;
    static constexpr int kWarpItems = 32 * 4 * VECS;
    static constexpr int kTile = NS_ * 32 * 4 * VECS;
    static constexpr size_t kValueBytes = static_cast<size_t>(kTile) * 4;
    static constexpr size_t kABytes = kValueBytes;
    static constexpr size_t kBBytes = kValueBytes;
    static constexpr bool kHasExtra = false;
    static constexpr int kParts = NS_;                  // one part per consume warp
    static constexpr bool kWarpIndependent = true;      // no barrier in consume()
    static constexpr int kWarpStage = kWarpItems + 4;   // words, 16-byte multiple
    static constexpr size_t kScratchBytes = static_cast<size_t>(NS_) * kWarpStage * 4;
    struct Args {
        const uint32_t *in;
        int32_t threshold;
        uint32_t *out;
        int32_t *count;
        size_t n;
        unsigned num_tiles;
        bool out_aligned;
        size_t capture_chunk = 0;            // nonzero: try the one-pass capture first (a cooperative launch)
        uint32_t *block_sums = nullptr;      // the capture's block totals (one word per block)
    };
    // the kernel first tries the one-pass capture (capture.cuh) and returns
    // when it wrote the result
    static constexpr bool kCapturing = true;
    __device__ static bool may_capture(const Args &a) { return a.capture_chunk != 0; }
    template <int NW, unsigned CAP>
    __device__ static bool capture(const Args &a, uint32_t *smem, DevState *st, unsigned spin_limit)
    {
        return capture_gt<NW, CAP>(a.in, a.threshold, a.out, a.count, a.n, a.capture_chunk, a.block_sums, st,
                                   spin_limit, smem);
    }
    __device__ static unsigned tile_len(const Args &a, unsigned t)
    {
        const size_t rem = a.n - static_cast<size_t>(t) * kTile;
        return rem < static_cast<size_t>(kTile) ? static_cast<unsigned>(rem) : static_cast<unsigned>(kTile);
    }
    __device__ static unsigned copied(const Args &a, unsigned t) { return tile_len(a, t) & ~3u; }
    __device__ static const void *a_src(const Args &a, unsigned t) { return a.in + static_cast<size_t>(t) * kTile; }
    __device__ static unsigned a_bytes(const Args &a, unsigned t) { return copied(a, t) * 4u; }
    __device__ static void prefetch_l2(const Args &a, unsigned t, uint64_t pol)
    {
        if (a_bytes(a, t) != 0) bulk_prefetch_l2(a_src(a, t), a_bytes(a, t), pol);
    }
    __device__ static void b_copies(const Args &a, unsigned t, const void **src, unsigned *bytes, unsigned *off)
    {
        src[0] = a_src(a, t);
        bytes[0] = a_bytes(a, t);
        off[0] = 0;
    }
    // pass A: the kept count of each consume warp's part, one warp reduction
    // per part (see CompactPolicy::reduce_parts)
    __device__ static void reduce_parts(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int,
                                        S &v, unsigned &, uint32_t *part)
    {
        static_assert(NS_ % NR_ == 0 && kWarpItems / 4 % 32 == 0, "whole parts per reduce warp");
        constexpr int PPW = NS_ / NR_, CH = kWarpItems / 4 / 32;   // parts per warp, 4-value chunks per lane
        const int lane = rtid & 31, rw = rtid >> 5;
        const unsigned cp = copied(a, t), len = tile_len(a, t);
        const size_t base = static_cast<size_t>(t) * kTile;
        const int32_t thr = a.threshold;
        const uint4 *b4 = reinterpret_cast<const uint4 *>(abuf);
        const uint32_t *b1 = reinterpret_cast<const uint32_t *>(abuf);
        unsigned c[PPW];
        if (len == static_cast<unsigned>(kTile)) {
#pragma unroll
            for (int i = 0; i < PPW; ++i) {
                c[i] = 0;
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const uint4 q = b4[(rw + i * NR_) * (kWarpItems / 4) + k * 32 + lane];
                    c[i] += __popc(greater_mask(q.x, q.y, q.z, q.w, thr));
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < PPW; ++i) {
                c[i] = 0;
                for (int k = 0; k < CH; ++k) {
                    const unsigned e = static_cast<unsigned>((rw + i * NR_) * kWarpItems + 4 * (k * 32 + lane));
                    for (unsigned j = 0; j < 4; ++j)
                        if (e + j < len)
                            c[i] += (static_cast<int32_t>(e + j < cp ? b1[e + j] : a.in[base + e + j]) > thr) ? 1u : 0u;
                }
            }
        }
        const unsigned mine = store_part_counts<PPW, NR_>(c, rw, lane, part);
        v = (lane == 0) ? mine : 0u;
    }
    __device__ static void after_reduce(const Args &, unsigned, unsigned) {}
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *, uint32_t *, int warp,
                                       int lane, Release &release)
    {
        const unsigned t = ct.tile;
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        const uint32_t *vals = reinterpret_cast<const uint32_t *>(ct.buf);
        const unsigned len = tile_len(a, t);
        const unsigned cp = copied(a, t);
        const int32_t thr = a.threshold;
        uint32_t x[VECS][4], keep[VECS];
        if (len == static_cast<unsigned>(kTile)) {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(vals + wbase);
#pragma unroll
            for (int q = 0; q < VECS; ++q) {
                const uint4 u = v4[q * 32 + lane];
                x[q][0] = u.x;
                x[q][1] = u.y;
                x[q][2] = u.z;
                x[q][3] = u.w;
                keep[q] = greater_mask(u.x, u.y, u.z, u.w, thr);
            }
        } else {
#pragma unroll
            for (int q = 0; q < VECS; ++q) {
                uint32_t m = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const unsigned e = static_cast<unsigned>(wbase + (q * 32 + lane) * 4 + j);
                    x[q][j] = (e < cp) ? vals[e] : ((e < len) ? a.in[base + e] : 0u);
                    if (e < len && static_cast<int32_t>(x[q][j]) > thr) m |= 1u << j;
                }
                keep[q] = m;
            }
        }
        const size_t g0 = static_cast<size_t>(ct.prefix) + ct.part_excl[warp];
        release();   // values in registers, offset read: the B buffer and the record are free
        uint32_t *stage = reinterpret_cast<uint32_t *>(ct.scratch) + warp * kWarpStage;
        compact_write_warp<VECS>(x, keep, g0, lane, stage, a.out, a.out_aligned, a.n);
        if (t == a.num_tiles - 1 && warp == 0 && lane == 0) *a.count = static_cast<int32_t>(ct.prefix + ct.aggregate);
        return 0;   // no warp-totals buffer used
    }
};

}  // namespace devscan
