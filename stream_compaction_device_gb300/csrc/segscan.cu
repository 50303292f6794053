// Segmented scan (sm_103a): a nonzero head flag heads[i] starts a new
// segment at i (element 0 always starts one) and every segment is scanned on
// its own.
//
// lpnh.cn "并行扫描 Scan/Prefix Sum" section 7.2 names the segmented scan as
// the building block for sparse data.  It is the plain scan of the pairs
// (h, v) under
//     (h1, v1) . (h2, v2) = (h1 | h2,  h2 ? v2 : v1 (+) v2),
// an associative operator, so every level of the plain scan carries over
// with pairs: threads fold their 4 elements, warps scan rows of pairs with
// shuffles, the block scans the warp pairs, and tiles chain through the
// decoupled look-back.  The look-back itself needs no pairs: a tile that
// contains a head publishes the fold since its last head as its inclusive
// prefix at once (nothing before that head can change it), so a look-back
// only ever folds the plain aggregates of head-free tiles and stops at the
// first tile with a head.  Two kernels, as for the plain scan:
//   * the persistent two-pass pipeline (pipeline_l2.cuh) for 16-byte
//     aligned data from 2^19 elements: pass A copies values and heads and
//     reduces each tile's pair, pass B applies the prefix;
//   * one tile per block with the one-level look-back for everything else.
// Traffic: 4 + 1 bytes read and 4 written per element.
#include <atomic>

#include "core.cuh"
#include "launch.h"
#include "pipeline_l2.cuh"

namespace devscan {
namespace {

// ---------------------------------------------------------------------------
// Pair algebra
// ---------------------------------------------------------------------------
// a then b: b's head cuts a off.
template <class Op>
__device__ __forceinline__ void seg_combine(const Op &op, typename Op::S av, unsigned ah, typename Op::S &bv,
                                            unsigned &bh)
{
    if (!bh) bv = op(av, bv);
    bh |= ah;
}

// Bit j of the result is set when byte j of w is nonzero.
__device__ __forceinline__ unsigned head_bits(uint32_t w)
{
    return ((w & 0x000000ffu) ? 1u : 0u) | ((w & 0x0000ff00u) ? 2u : 0u) | ((w & 0x00ff0000u) ? 4u : 0u) |
           ((w & 0xff000000u) ? 8u : 0u);
}

// Fold of one thread-row of 4 elements with head bits hb: (any head, fold
// since the last head).
template <class Op>
__device__ __forceinline__ void seg_fold4(const Op &op, const typename Op::S (&x)[4], unsigned hb,
                                          typename Op::S &v, unsigned &h)
{
    v = Op::identity();
#pragma unroll
    for (int j = 0; j < 4; ++j) v = ((hb >> j) & 1u) ? x[j] : op(v, x[j]);
    h = hb != 0 ? 1u : 0u;
}

// Warp level, VECS rows of 32 lanes (row-major: row r, then lane): exclusive
// pair of every lane-row and the warp's total pair.
template <class Op, int VECS>
__device__ __forceinline__ void seg_warp_scan_rows(const Op &op, const typename Op::S (&tv)[VECS],
                                                   const unsigned (&th)[VECS], int lane, typename Op::S (&ev)[VECS],
                                                   unsigned (&eh)[VECS], typename Op::S &wv, unsigned &wh)
{
    using S = typename Op::S;
    S iv[VECS];
    unsigned ih[VECS];
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        iv[r] = tv[r];
        ih[r] = th[r];
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            const S uv = __shfl_up_sync(kFullMask, iv[r], d);
            const unsigned uh = __shfl_up_sync(kFullMask, ih[r], d);
            if (lane >= d) seg_combine(op, uv, uh, iv[r], ih[r]);
        }
    }
    S rv = Op::identity();
    unsigned rh = 0;
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        S bv = __shfl_up_sync(kFullMask, iv[r], 1);
        unsigned bh = __shfl_up_sync(kFullMask, ih[r], 1);
        if (lane == 0) {
            bv = Op::identity();
            bh = 0;
        }
        seg_combine(op, rv, rh, bv, bh);
        ev[r] = bv;
        eh[r] = bh;
        S tv31 = __shfl_sync(kFullMask, iv[r], 31);
        unsigned th31 = __shfl_sync(kFullMask, ih[r], 31);
        seg_combine(op, rv, rh, tv31, th31);
        rv = tv31;
        rh = th31;
    }
    wv = rv;
    wh = rh;
}

// Block level: NW warp pairs in shared memory (values in bv, heads in bh),
// already written and made visible by the caller's barrier; every warp
// scans them and takes its exclusive pair and the block total.
template <class Op, int NW>
__device__ __forceinline__ void seg_scan_warp_pairs(const Op &op, const uint32_t *bv, const uint32_t *bh, int warp,
                                                    int lane, typename Op::S &xv, unsigned &xh,
                                                    typename Op::S &tv, unsigned &th)
{
    using S = typename Op::S;
    S v = (lane < NW) ? from_bits<S>(bv[lane]) : Op::identity();
    unsigned h = (lane < NW) ? bh[lane] : 0u;
#pragma unroll
    for (int d = 1; d < NW; d <<= 1) {
        const S uv = __shfl_up_sync(kFullMask, v, d);
        const unsigned uh = __shfl_up_sync(kFullMask, h, d);
        if (lane >= d) seg_combine(op, uv, uh, v, h);
    }
    const S pv = __shfl_sync(kFullMask, v, warp > 0 ? warp - 1 : 0);
    const unsigned ph = __shfl_sync(kFullMask, h, warp > 0 ? warp - 1 : 0);
    xv = (warp > 0) ? pv : Op::identity();
    xh = (warp > 0) ? ph : 0u;
    tv = __shfl_sync(kFullMask, v, NW - 1);
    th = __shfl_sync(kFullMask, h, NW - 1);
}

// Applies the carry c (the fold of everything before this warp's part) and
// scans the rows in place.  ev/eh: exclusive pairs of the lane-rows within
// the warp; (xv, xh): the warp's exclusive pair within the tile.
template <class Op, bool INCLUSIVE, int VECS>
__device__ __forceinline__ void seg_finish_rows(const Op &op, typename Op::S carry, typename Op::S xv, unsigned xh,
                                                const typename Op::S (&ev)[VECS], const unsigned (&eh)[VECS],
                                                const unsigned (&hb)[VECS], typename Op::S (&x)[VECS][4])
{
    using S = typename Op::S;
    const S wcarry = xh ? xv : op(carry, xv);
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        S cur = eh[r] ? ev[r] : op(wcarry, ev[r]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if ((hb[r] >> j) & 1u) cur = Op::identity();
            const S v = x[r][j];
            if (INCLUSIVE) {
                cur = op(cur, v);
                x[r][j] = cur;
            } else {
                x[r][j] = cur;
                cur = op(cur, v);
            }
        }
    }
}

// Head bits of this thread's rows: bit j of hb[r] is the head flag of
// element (r * 32 + lane) * 4 + j of the warp's part (0 past n).
template <int VECS, bool ALIGNED>
__device__ __forceinline__ void load_head_rows(const uint8_t *__restrict__ heads, size_t warp_base, size_t n,
                                               int lane, bool full, unsigned (&hb)[VECS])
{
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        const size_t e = warp_base + static_cast<size_t>(r * 32 + lane) * 4;
        if (ALIGNED && full) {
            hb[r] = head_bits(__ldcs(reinterpret_cast<const uint32_t *>(heads + e)));
        } else {
            unsigned m = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (e + j < n && heads[e + j] != 0) m |= 1u << j;
            hb[r] = m;
        }
    }
}

// ---------------------------------------------------------------------------
// One tile per block (tickets in launch order), one-level look-back.
// ALIGNED: values 16-byte and heads 4-byte aligned.
// ---------------------------------------------------------------------------
template <class Op, int THREADS, int VECS, bool INCLUSIVE, bool ALIGNED>
__global__ void __launch_bounds__(THREADS)
segscan_tile_kernel(const typename Op::S *__restrict__ in, const uint8_t *__restrict__ heads,
                    typename Op::S *__restrict__ out, size_t n, unsigned num_tiles, unsigned long long *status,
                    DevState *st, unsigned capacity, unsigned spin_limit)
{
    using S = typename Op::S;
    constexpr int NWARPS = THREADS / 32;
    constexpr int WARP_ITEMS = 32 * 4 * VECS;
    constexpr int TILE = THREADS * 4 * VECS;
    __shared__ uint32_t s_wv[NWARPS], s_wh[NWARPS];
    __shared__ uint32_t s_prefix;
    __shared__ unsigned s_tile, s_tag;
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // The epoch is read before the ticket is taken (the fence orders the
    // two).  A tile with a head publishes its inclusive prefix without
    // waiting for its predecessors, so the last tile's look-back -- after
    // which its block closes the launch and advances the epoch -- can end
    // while earlier blocks are still starting; each of them must already
    // hold the launch's epoch by then, and every ticket has been taken.
    if (tid == 0) {
        s_tag = read_tag(st);
        __threadfence();
        s_tile = atomicAdd(&st->ticket, 1u);
    }
    __syncthreads();
    const unsigned tile = s_tile;
    if (tile >= num_tiles) return;   // never taken: each launch hands out exactly num_tiles tickets
    const size_t tile_base = static_cast<size_t>(tile) * TILE;
    const size_t warp_base = tile_base + static_cast<size_t>(warp) * WARP_ITEMS;
    const bool full = tile_base + TILE <= n;

    S x[VECS][4];
    unsigned hb[VECS];
    load_rows<S, VECS, ALIGNED>(in, warp_base, n, lane, full, x, Op::identity());
    load_head_rows<VECS, ALIGNED>(heads, warp_base, n, lane, full, hb);

    S tv[VECS], ev[VECS], wv;
    unsigned th[VECS], eh[VECS], wh;
#pragma unroll
    for (int r = 0; r < VECS; ++r) seg_fold4<Op>(op, x[r], hb[r], tv[r], th[r]);
    seg_warp_scan_rows<Op, VECS>(op, tv, th, lane, ev, eh, wv, wh);
    if (lane == 0) {
        s_wv[warp] = to_bits(wv);
        s_wh[warp] = wh;
    }
    __syncthreads();
    S xv, totv;
    unsigned xh, toth;
    seg_scan_warp_pairs<Op, NWARPS>(op, s_wv, s_wh, warp, lane, xv, xh, totv, toth);

    if (warp == 0) {
        const unsigned tag = s_tag;
        // a tile with a head knows its inclusive prefix already
        publish<Op>(status, tile, tag, (tile == 0 || toth) ? kFlagInclusive : kFlagAggregate, totv, lane);
        S prefix = Op::identity();
        if (tile != 0) {
            prefix = lookback<Op, kLookbackPerLane>(op, status, tile, tag, &st->error, spin_limit, lane);
            if (!toth) publish<Op>(status, tile, tag, kFlagInclusive, op(prefix, totv), lane);
        }
        if (lane == 0) s_prefix = to_bits(prefix);
        if (tile == num_tiles - 1) finish_launch(st, status, num_tiles, capacity, lane);
    }
    __syncthreads();

    seg_finish_rows<Op, INCLUSIVE, VECS>(op, from_bits<S>(s_prefix), xv, xh, ev, eh, hb, x);
    store_rows<S, VECS, ALIGNED>(out, warp_base, n, lane, full, x);
}

// Index of the highest nonzero byte of a nonzero word.
__device__ __forceinline__ int top_byte(uint32_t w) { return (31 - __clz(static_cast<int>(w))) >> 3; }

// ---------------------------------------------------------------------------
// Pipelined policy (see pipeline_l2.cuh).  Both passes copy the tile's values
// (kTile * 4 bytes) followed by its heads (kTile bytes).  The tile splits into
// one part per consume warp; a reduce warp takes whole parts: it finds a
// part's last head (a warp max) and folds the values from it on, so that fold
// needs no order, and reports the part's (head, value) pair.  The kernel folds
// the pairs in order into the tile's pair, and every consume warp combines the
// pairs of the parts before its own with the tile's prefix -- no barrier
// among the consume warps.
// ---------------------------------------------------------------------------
template <class OpT, bool INCLUSIVE, int NS_, int NR_, int VECS_, int SA_, int SB_, int R_, int PREFETCH = 0>
struct SegScanPolicy {
    using Op = OpT;
    using S = typename Op::S;
    static constexpr bool kSegmented = true;
    static constexpr int kAHint = kL2EvictLast, kBHint = kL2EvictFirst, kPrefetch = PREFETCH;
    static constexpr int kConsumeWarps = NS_, kReduceWarps = NR_, kRecords = R_, kAStages = SA_, kBStages = SB_;
    static constexpr int VECS = VECS_;
    static constexpr int kWarpItems = 32 * 4 * VECS;
    static constexpr int kTile = NS_ * 32 * 4 * VECS;
    static constexpr size_t kValueBytes = static_cast<size_t>(kTile) * 4;
    static constexpr size_t kABytes = kValueBytes + static_cast<size_t>(kTile);
    static constexpr size_t kBBytes = kABytes;
    static constexpr int kParts = NS_;                   // one part per consume warp
    static constexpr bool kWarpIndependent = true;       // no barrier in consume()
    static constexpr bool kHasExtra = false;
    struct Args {
        const S *in;
        const uint8_t *heads;
        S *out;
        size_t n;
    };
    __device__ static unsigned tile_len(const Args &a, unsigned t)
    {
        const size_t rem = a.n - static_cast<size_t>(t) * kTile;
        return rem < static_cast<size_t>(kTile) ? static_cast<unsigned>(rem) : static_cast<unsigned>(kTile);
    }
    __device__ static unsigned values_copied(const Args &a, unsigned t) { return tile_len(a, t) & ~3u; }
    __device__ static unsigned heads_copied(const Args &a, unsigned t) { return tile_len(a, t) & ~15u; }
    __device__ static void a_copies(const Args &a, unsigned t, const void **src, unsigned *bytes, unsigned *off)
    {
        src[0] = a.in + static_cast<size_t>(t) * kTile;
        bytes[0] = values_copied(a, t) * 4u;
        off[0] = 0;
        src[1] = a.heads + static_cast<size_t>(t) * kTile;
        bytes[1] = heads_copied(a, t);
        off[1] = static_cast<unsigned>(kValueBytes);
    }
    // unused (a_copies replaces them); kept for the interface
    __device__ static const void *a_src(const Args &a, unsigned t) { return a.in + static_cast<size_t>(t) * kTile; }
    __device__ static unsigned a_bytes(const Args &a, unsigned t) { return values_copied(a, t) * 4u; }
    __device__ static void prefetch_l2(const Args &a, unsigned t, uint64_t pol)
    {
        if (values_copied(a, t) != 0)
            bulk_prefetch_l2(a.in + static_cast<size_t>(t) * kTile, values_copied(a, t) * 4u, pol);
        if (heads_copied(a, t) != 0) bulk_prefetch_l2(a.heads + static_cast<size_t>(t) * kTile, heads_copied(a, t), pol);
    }
    __device__ static void b_copies(const Args &a, unsigned t, const void **src, unsigned *bytes, unsigned *off)
    {
        a_copies(a, t, src, bytes, off);
    }
    // pass A: each part's pair -- value in part[q], head flag in
    // part[kParts + q]; reduce warp rw takes parts rw, rw + NR, ...
    __device__ static void reduce_parts(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int, S &v,
                                        unsigned &extra, uint32_t *part)
    {
        static_assert(NS_ % NR_ == 0 && kWarpItems == 512, "whole parts of 16 heads per lane");
        const Op op;
        const int lane = rtid & 31, rw = rtid >> 5;
        const unsigned len = tile_len(a, t);
        const unsigned vcp = values_copied(a, t), hcp = heads_copied(a, t);
        const size_t base = static_cast<size_t>(t) * kTile;
        const S *vals = reinterpret_cast<const S *>(abuf);
        const uint8_t *hd = abuf + kValueBytes;
        v = Op::identity();
        extra = 0;
#pragma unroll
        for (int i = 0; i < NS_ / NR_; ++i) {
            const int q = rw + i * NR_;
            const unsigned p0 = static_cast<unsigned>(q) * kWarpItems;
            const unsigned p1 = (p0 + kWarpItems < len) ? p0 + kWarpItems : (p0 < len ? len : p0);
            // last head of the part (-1: none); lane L looks at heads 16L .. 16L + 15
            int last = -1;
            if (p1 == p0 + kWarpItems && p1 <= hcp) {
                const uint4 h = reinterpret_cast<const uint4 *>(hd + p0)[lane];
                const int at = static_cast<int>(p0) + lane * 16;
                if (h.w) last = at + 12 + top_byte(h.w);
                else if (h.z) last = at + 8 + top_byte(h.z);
                else if (h.y) last = at + 4 + top_byte(h.y);
                else if (h.x) last = at + top_byte(h.x);
            } else {
                for (unsigned e = p0 + 16u * lane; e < p0 + 16u * lane + 16u && e < p1; ++e) {
                    const uint8_t h = (e < hcp) ? hd[e] : a.heads[base + e];
                    if (h != 0) last = static_cast<int>(e);
                }
            }
            last = __reduce_max_sync(kFullMask, last);
            const unsigned from = last >= 0 ? static_cast<unsigned>(last) : p0;
            S pv = Op::identity();
            if (p1 == p0 + kWarpItems && p1 <= vcp) {
                // lane L takes the 16-byte groups L, L + 32, L + 64, L + 96
                const uint4 *v4 = reinterpret_cast<const uint4 *>(vals + p0);
                const S id = Op::identity();
#pragma unroll
                for (int g = 0; g < kWarpItems / 128; ++g) {
                    const unsigned e = p0 + 4u * static_cast<unsigned>(g * 32 + lane);
                    const uint4 u = v4[g * 32 + lane];
                    pv = op(pv, op(op(e >= from ? from_bits<S>(u.x) : id, e + 1 >= from ? from_bits<S>(u.y) : id),
                                   op(e + 2 >= from ? from_bits<S>(u.z) : id, e + 3 >= from ? from_bits<S>(u.w) : id)));
                }
            } else {
                for (unsigned e = from + lane; e < p1; e += 32) pv = op(pv, (e < vcp) ? vals[e] : a.in[base + e]);
            }
            pv = warp_fold(op, pv);
            if (lane == 0) {
                part[q] = to_bits(pv);
                part[kParts + q] = last >= 0 ? 1u : 0u;
            }
        }
    }
    __device__ static void after_reduce(const Args &, unsigned, unsigned) {}
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *, uint32_t *,
                                       int warp, int lane, Release &release)
    {
        const Op op;
        const unsigned t = ct.tile;
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        const S *vals = reinterpret_cast<const S *>(ct.buf);
        const uint8_t *hd = ct.buf + kValueBytes;
        const unsigned len = tile_len(a, t);
        S x[VECS][4];
        unsigned hb[VECS];
        if (len == static_cast<unsigned>(kTile)) {
            const uint4 *v4 = reinterpret_cast<const uint4 *>(vals + wbase);
            const uint32_t *h32 = reinterpret_cast<const uint32_t *>(hd + wbase);
#pragma unroll
            for (int q = 0; q < VECS; ++q) {
                const uint4 u = v4[q * 32 + lane];
                x[q][0] = from_bits<S>(u.x);
                x[q][1] = from_bits<S>(u.y);
                x[q][2] = from_bits<S>(u.z);
                x[q][3] = from_bits<S>(u.w);
                hb[q] = head_bits(h32[q * 32 + lane]);
            }
        } else {
            const unsigned vcp = values_copied(a, t), hcp = heads_copied(a, t);
#pragma unroll
            for (int q = 0; q < VECS; ++q) {
                unsigned m = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const unsigned e = static_cast<unsigned>(wbase + (q * 32 + lane) * 4 + j);
                    x[q][j] = (e < vcp) ? vals[e] : ((e < len) ? a.in[base + e] : Op::identity());
                    const uint8_t h = (e < hcp) ? hd[e] : ((e < len) ? a.heads[base + e] : uint8_t(0));
                    if (h != 0) m |= 1u << j;
                }
                hb[q] = m;
            }
        }
        // this warp's exclusive pair within the tile: lane q < kParts holds
        // part q's pair; an in-order pair scan, then lane warp - 1's result
        S pv = lane < kParts ? from_bits<S>(ct.part_excl[lane]) : Op::identity();
        unsigned ph = lane < kParts ? (ct.part_excl[kParts] >> lane) & 1u : 0u;
        release();   // the tile and the part pairs are in registers now
#pragma unroll
        for (int d = 1; d < kParts; d <<= 1) {
            const S uv = __shfl_up_sync(kFullMask, pv, d);
            const unsigned uh = __shfl_up_sync(kFullMask, ph, d);
            if (lane >= d) seg_combine(op, uv, uh, pv, ph);
        }
        S xv = __shfl_sync(kFullMask, pv, warp > 0 ? warp - 1 : 0);
        unsigned xh = __shfl_sync(kFullMask, ph, warp > 0 ? warp - 1 : 0);
        if (warp == 0) {
            xv = Op::identity();
            xh = 0;
        }
        S tv[VECS], ev[VECS], wv;
        unsigned th[VECS], eh[VECS], wh;
#pragma unroll
        for (int q = 0; q < VECS; ++q) seg_fold4<Op>(op, x[q], hb[q], tv[q], th[q]);
        seg_warp_scan_rows<Op, VECS>(op, tv, th, lane, ev, eh, wv, wh);
        seg_finish_rows<Op, INCLUSIVE, VECS>(op, ct.prefix, xv, xh, ev, eh, hb, x);
        if (base + kTile <= a.n) {
            uint4 *o4 = reinterpret_cast<uint4 *>(a.out + base + wbase);
#pragma unroll
            for (int q = 0; q < VECS; ++q)
                st_stream(o4 + q * 32 + lane,
                          make_uint4(to_bits(x[q][0]), to_bits(x[q][1]), to_bits(x[q][2]), to_bits(x[q][3])));
        } else {
#pragma unroll
            for (int q = 0; q < VECS; ++q)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const size_t e = base + wbase + static_cast<size_t>((q * 32 + lane) * 4 + j);
                    if (e < a.n) a.out[e] = x[q][j];
                }
        }
        return 0;   // no warp-totals buffer used
    }
};

constexpr unsigned kSegWaitLimit = 1u << 18;
constexpr size_t kSegPipelineMinN = size_t(1) << 19;

template <class Op, bool INCLUSIVE>
cudaError_t launch_seg_pipelined(const void *in, const uint8_t *heads, void *out, size_t n, const Workspace &ws,
                                 unsigned spin_limit, cudaStream_t s)
{
    using S = typename Op::S;
    // eight reduce warps (two parts each) and six records: measured at 2^28,
    // 424 us against 532 us with four reduce warps and ten records -- the
    // reduce step, not the records, bounds the tile rate
    using P = SegScanPolicy<Op, INCLUSIVE, 16, 8, 4, 3, 2, 6, 1>;
    using G = PipeShape<P>;
    auto kernel = pipeline_l2_kernel<P>;
    static std::atomic<unsigned long long> attribute_set{0};   // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if ((attribute_set.load() & bit) == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(G::kSmemBytes));
        if (e != cudaSuccess) return e;
        attribute_set.fetch_or(bit);
    }
    const unsigned tiles = tiles_for(n, P::kTile);
    const unsigned grid = tiles < static_cast<unsigned>(ws.num_sms) ? tiles : static_cast<unsigned>(ws.num_sms);
    typename P::Args args{static_cast<const S *>(in), heads, static_cast<S *>(out), n};
    kernel<<<grid, G::kThreads, G::kSmemBytes, s>>>(args, tiles, ws.status, ws.state, ws.capacity, spin_limit,
                                                    kSegWaitLimit);
    return cudaGetLastError();
}

template <class Op, bool INCLUSIVE>
cudaError_t launch_seg(const void *in, const uint8_t *heads, void *out, size_t n, int carry, const Workspace &ws,
                       unsigned spin_limit, cudaStream_t s)
{
    using S = typename Op::S;
    const uintptr_t pi = reinterpret_cast<uintptr_t>(in), po = reinterpret_cast<uintptr_t>(out),
                    ph = reinterpret_cast<uintptr_t>(heads);
    const bool bulk_ok = pi % 16 == 0 && po % 16 == 0 && ph % 16 == 0;
    if (bulk_ok && (carry == kCarryPipelined || (carry != kCarryLookback && n >= kSegPipelineMinN)))
        return launch_seg_pipelined<Op, INCLUSIVE>(in, heads, out, n, ws, spin_limit, s);
    const unsigned tiles = tiles_for(n, kScanTile);
    const S *sin = static_cast<const S *>(in);
    S *sout = static_cast<S *>(out);
    if (pi % 16 == 0 && po % 16 == 0 && ph % 4 == 0)
        segscan_tile_kernel<Op, kScanThreads, kScanVecs, INCLUSIVE, true><<<tiles, kScanThreads, 0, s>>>(
            sin, heads, sout, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    else
        segscan_tile_kernel<Op, kScanThreads, kScanVecs, INCLUSIVE, false><<<tiles, kScanThreads, 0, s>>>(
            sin, heads, sout, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    return cudaGetLastError();
}

template <class Op>
cudaError_t launch_seg_dir(bool inclusive, const void *in, const uint8_t *heads, void *out, size_t n, int carry,
                           const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    return inclusive ? launch_seg<Op, true>(in, heads, out, n, carry, ws, spin_limit, s)
                     : launch_seg<Op, false>(in, heads, out, n, carry, ws, spin_limit, s);
}

}  // namespace

cudaError_t launch_segscan(ElemType type, int op, bool inclusive, const void *in, const uint8_t *heads, void *out,
                           size_t n, int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    switch (type) {
    case ElemType::I32:
        if (op == kOpAdd) return launch_seg_dir<AddU32>(inclusive, in, heads, out, n, carry, ws, spin_limit, s);
        if (op == kOpMax) return launch_seg_dir<MaxI32>(inclusive, in, heads, out, n, carry, ws, spin_limit, s);
        return launch_seg_dir<XorU32>(inclusive, in, heads, out, n, carry, ws, spin_limit, s);
    case ElemType::U32:
        if (op == kOpAdd) return launch_seg_dir<AddU32>(inclusive, in, heads, out, n, carry, ws, spin_limit, s);
        if (op == kOpMax) return launch_seg_dir<MaxU32>(inclusive, in, heads, out, n, carry, ws, spin_limit, s);
        return launch_seg_dir<XorU32>(inclusive, in, heads, out, n, carry, ws, spin_limit, s);
    case ElemType::F32:
        if (op == kOpAdd) return launch_seg_dir<AddF32>(inclusive, in, heads, out, n, carry, ws, spin_limit, s);
        return launch_seg_dir<MaxF32>(inclusive, in, heads, out, n, carry, ws, spin_limit, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace devscan
