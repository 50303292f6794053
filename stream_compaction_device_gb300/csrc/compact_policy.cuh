// Compaction policy of the persistent two-pass pipeline (sm_103a), and the
// byte-flag helpers both compaction kernels use.
#pragma once

#include "core.cuh"
#include "pipeline_l2.cuh"
#include "stage.cuh"

namespace devscan {

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t *p) { return __ldcs(p); }

// Bit k set when byte k of f is nonzero.
__device__ __forceinline__ uint32_t nonzero_byte_mask(uint32_t f)
{
    return ((f & 0x000000ffu) ? 1u : 0u) | ((f & 0x0000ff00u) ? 2u : 0u) | ((f & 0x00ff0000u) ? 4u : 0u) |
           ((f & 0xff000000u) ? 8u : 0u);
}

// ---------------------------------------------------------------------------
// Pipelined compaction (see pipeline_l2.cuh): pass A reads only the tile's
// flags (1 byte per element) and counts the kept elements -- the aggregate
// the look-back carries; pass B reads the values and (from L2) the flags,
// ranks the kept values, stages them in the B buffer at their tile rank and
// writes one contiguous run at the tile's prefix.  HBM traffic is the
// algorithmic 5 bytes per element plus 4 per kept element.
// ---------------------------------------------------------------------------
constexpr unsigned kBarCompactStage = 8;

// Second half of a compaction consume step, shared by both predicate forms:
// ranks the kept elements (bit j of keep[q] keeps x[q][j]), stages them in
// `stage` in phase with their destination (so the copy out is straight
// 128-bit chunks; `stage` must hold the tile plus 3 words and must be free to
// overwrite once the group scan's barrier has passed) and writes them as one
// contiguous run at the tile's prefix.  The last tile also writes the count.
template <int NS, int VECS>
__device__ __forceinline__ void compact_write_tile(const uint32_t (&x)[VECS][4], const uint32_t (&keep)[VECS],
                                                   const ConsumeTile<uint32_t> &ct, uint32_t *wbuf0, uint32_t *wbuf1,
                                                   int warp, int lane, uint32_t *stage, uint32_t *out,
                                                   bool out_aligned, size_t n, int32_t *count, bool last_tile)
{
    constexpr int THREADS = NS * 32;
    const AddU32 op;
    uint32_t cnt[VECS];
#pragma unroll
    for (int q = 0; q < VECS; ++q) cnt[q] = __popc(keep[q]);
    uint32_t row_excl[VECS], warp_total;
    warp_scan_rows<AddU32, VECS>(op, cnt, lane, row_excl, warp_total);
    uint32_t warp_excl, total;
    // the barrier inside also means every thread has read the buffer
    group_scan<AddU32, NS>(op, warp_total, (ct.round & 1) ? wbuf1 : wbuf0, warp, lane, warp_excl, total);
    const unsigned phase = out_aligned ? (ct.prefix & 3u) : 0u;
#pragma unroll
    for (int q = 0; q < VECS; ++q) {
        uint32_t rank = phase + warp_excl + row_excl[q];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if ((keep[q] >> j) & 1u) stage[rank++] = x[q][j];
    }
    named_sync(kBarCompactStage, THREADS);
    const unsigned tid = static_cast<unsigned>(warp * 32 + lane);
    if (out_aligned)
        write_run_direct<THREADS>(out, ct.prefix, total, stage, static_cast<int>(tid), n);
    else
        write_run_scalar<THREADS>(out, ct.prefix, total, stage, 0, static_cast<int>(tid), n);
    if (last_tile && tid == 0) *count = static_cast<int32_t>(ct.prefix + total);
}

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
    // both arrays: pass B then finds the values in L2 as well
    __device__ static void prefetch_l2(const Args &a, unsigned t, uint64_t pol)
    {
        if (flags_copied(a, t) != 0) bulk_prefetch_l2(a_src(a, t), flags_copied(a, t), pol);
        if (values_copied(a, t) != 0)
            bulk_prefetch_l2(a.in + static_cast<size_t>(t) * kTile, values_copied(a, t) * 4u, pol);
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
    __device__ static void reduce(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int nthr, S &v,
                                  unsigned &)
    {
        const unsigned cp = flags_copied(a, t);
        unsigned c = 0;
        const uint4 *f4 = reinterpret_cast<const uint4 *>(abuf);
        for (unsigned k = rtid; k < cp / 16; k += nthr) {
            const uint4 q = f4[k];
            c += __popc(nonzero_byte_mask(q.x)) + __popc(nonzero_byte_mask(q.y)) + __popc(nonzero_byte_mask(q.z)) +
                 __popc(nonzero_byte_mask(q.w));
        }
        const size_t base = static_cast<size_t>(t) * kTile;
        const unsigned len = tile_len(a, t);
        for (unsigned e = cp + rtid; e < len; e += nthr) c += a.flags[base + e] != 0 ? 1u : 0u;
        v = c;
    }
    __device__ static void after_reduce(const Args &, unsigned, unsigned) {}
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *wbuf0, uint32_t *wbuf1,
                                       int warp, int lane, Release &release)
    {
        const unsigned t = ct.tile;
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        uint32_t *vals = reinterpret_cast<uint32_t *>(ct.buf);
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
        // the staged run may run three words into the flags area, which is
        // read already
        compact_write_tile<NS_, VECS>(x, keep, ct, wbuf0, wbuf1, warp, lane, vals, a.out, a.out_aligned, a.n, a.count,
                                      t == a.num_tiles - 1);
        release();
        return 1;
    }
};

// Keep mask of four int32 values against a threshold: bit j set when
// (int32) v_j > t.
__device__ __forceinline__ uint32_t greater_mask(uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3, int32_t t)
{
    return (static_cast<int32_t>(v0) > t ? 1u : 0u) | (static_cast<int32_t>(v1) > t ? 2u : 0u) |
           (static_cast<int32_t>(v2) > t ? 4u : 0u) | (static_cast<int32_t>(v3) > t ? 8u : 0u);
}

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
    static constexpr size_t kBBytes = kValueBytes + 16;   // + room for the staging phase (3 words)
    static constexpr bool kHasExtra = false;
    struct Args {
        const uint32_t *in;
        int32_t threshold;
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
    __device__ static void reduce(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int nthr, S &v,
                                  unsigned &)
    {
        const unsigned cp = copied(a, t);
        const int32_t thr = a.threshold;
        unsigned c = 0;
        const uint4 *b4 = reinterpret_cast<const uint4 *>(abuf);
#pragma unroll 4
        for (unsigned k = rtid; k < cp / 4; k += nthr) {
            const uint4 q = b4[k];
            c += __popc(greater_mask(q.x, q.y, q.z, q.w, thr));
        }
        const size_t base = static_cast<size_t>(t) * kTile;
        const unsigned len = tile_len(a, t);
        for (unsigned e = cp + rtid; e < len; e += nthr) c += static_cast<int32_t>(a.in[base + e]) > thr ? 1u : 0u;
        v = c;
    }
    __device__ static void after_reduce(const Args &, unsigned, unsigned) {}
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *wbuf0, uint32_t *wbuf1,
                                       int warp, int lane, Release &release)
    {
        const unsigned t = ct.tile;
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        uint32_t *vals = reinterpret_cast<uint32_t *>(ct.buf);
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
        compact_write_tile<NS_, VECS>(x, keep, ct, wbuf0, wbuf1, warp, lane, vals, a.out, a.out_aligned, a.n, a.count,
                                      t == a.num_tiles - 1);
        release();
        return 1;
    }
};

}  // namespace devscan
