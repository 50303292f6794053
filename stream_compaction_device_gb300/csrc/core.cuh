// Device building blocks of the single-pass scan, compaction and split
// kernels for sm_103a.
//
// Data layout of one tile (THREADS threads, VECS 16-byte rows per thread):
// warp w owns a contiguous run of 32 * 4 * VECS elements; in row r, lane l
// holds the four consecutive elements of 16-byte chunk (r * 32 + l) of that
// run.  Every load and store instruction of a warp therefore touches 512
// contiguous bytes (coalesced, 128-bit per thread), and the run's order is
// row-major: row 0 of all lanes, then row 1, and so on.
//
// Scan levels (geek-doc.cn "并行前缀和 scan ..." sections 一, 四, 五):
//   thread : serial combine of its 4 elements of a row;
//   warp   : shuffle-up scan of the 32 lane totals of a row (5 steps, with the
//            lane >= delta guard), rows chained by their warp totals;
//   block  : warp totals through shared memory, scanned by every warp;
//   device : single-pass chained scan -- each tile publishes its aggregate,
//            then looks back over its predecessors' status words for the
//            nearest inclusive prefix (the inter-block carry).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace devscan {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// Associative operators.  S is the element type in registers and memory.
// Integer add and xor work on uint32_t (int32 add wraps modulo 2^32 exactly
// like uint32 add, so both share the same kernel).
// ---------------------------------------------------------------------------
struct AddU32 {
    using S = uint32_t;
    static __device__ __forceinline__ S identity() { return 0u; }
    __device__ __forceinline__ S operator()(S a, S b) const { return a + b; }
};
struct XorU32 {
    using S = uint32_t;
    static __device__ __forceinline__ S identity() { return 0u; }
    __device__ __forceinline__ S operator()(S a, S b) const { return a ^ b; }
};
struct MaxU32 {
    using S = uint32_t;
    static __device__ __forceinline__ S identity() { return 0u; }
    __device__ __forceinline__ S operator()(S a, S b) const { return a >= b ? a : b; }
};
struct MaxI32 {
    using S = int32_t;
    static __device__ __forceinline__ S identity() { return INT32_MIN; }
    __device__ __forceinline__ S operator()(S a, S b) const { return a >= b ? a : b; }
};
struct AddF32 {
    using S = float;
    static __device__ __forceinline__ S identity() { return 0.0f; }
    __device__ __forceinline__ S operator()(S a, S b) const { return __fadd_rn(a, b); }
};
struct MaxF32 {
    using S = float;
    static __device__ __forceinline__ S identity() { return -__int_as_float(0x7f800000); }
    __device__ __forceinline__ S operator()(S a, S b) const { return fmaxf(a, b); }
};

// Fold of v over the warp (the result in every lane): one redux instruction
// for the integer operators, shuffles for fp32.
__device__ __forceinline__ uint32_t warp_fold(const AddU32 &, uint32_t v) { return __reduce_add_sync(kFullMask, v); }
__device__ __forceinline__ uint32_t warp_fold(const XorU32 &, uint32_t v) { return __reduce_xor_sync(kFullMask, v); }
__device__ __forceinline__ uint32_t warp_fold(const MaxU32 &, uint32_t v) { return __reduce_max_sync(kFullMask, v); }
__device__ __forceinline__ int32_t warp_fold(const MaxI32 &, int32_t v) { return __reduce_max_sync(kFullMask, v); }
template <class Op>
__device__ __forceinline__ typename Op::S warp_fold(const Op &op, typename Op::S v)
{
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
    return v;
}

__device__ __forceinline__ uint32_t to_bits(uint32_t v) { return v; }
__device__ __forceinline__ uint32_t to_bits(int32_t v) { return static_cast<uint32_t>(v); }
__device__ __forceinline__ uint32_t to_bits(float v) { return __float_as_uint(v); }

template <typename S> __device__ __forceinline__ S from_bits(uint32_t b);
template <> __device__ __forceinline__ uint32_t from_bits<uint32_t>(uint32_t b) { return b; }
template <> __device__ __forceinline__ int32_t from_bits<int32_t>(uint32_t b) { return static_cast<int32_t>(b); }
template <> __device__ __forceinline__ float from_bits<float>(uint32_t b) { return __uint_as_float(b); }

// ---------------------------------------------------------------------------
// Per-stream device state (lives at the start of the workspace).
//   epoch  : stored as tag - 1; status words carry the tag of the launch that
//            wrote them, so words of earlier launches read as "not ready"
//            and the status array never needs clearing between launches.
//            The launch that owns the last tile advances it.
//   ticket : next tile index handed out (dynamic tile order); the last
//            tile's block resets it to 0 for the next launch.
//   error  : sticky device error bits, read and cleared by the host.
//   cursor : rolling position for refreshing status slots that recent
//            launches did not use (so no stale word outlives 2^30 epochs).
//   zeros  : zero counts per bit for the split / radix sort.
//   capture_abort / capture_wait : the fused-predicate compaction's
//            one-pass capture, and the back-off after a capture gave up.
// ---------------------------------------------------------------------------
struct DevState {
    unsigned epoch;
    unsigned ticket;
    unsigned error;
    unsigned cursor;
    unsigned grid_arrive;   // blocks that reached the grid barrier, or that handed in their totals
                            // (the last one of those resets it)
    unsigned grid_depart;   // blocks that left it; the last one resets both
    unsigned capture_abort; // a fused-predicate capture gave up (reset by its last block to leave)
    unsigned capture_wait;  // calls still to skip the capture after one gave up (a back-off)
    unsigned pad[8];
    unsigned zeros[48];
};
static_assert(sizeof(DevState) == 256, "DevState is 256 bytes in every workspace layout");

constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kEpochTags = (1u << 30) - 1u;   // tags 1 .. 2^30 - 1
constexpr unsigned kRefreshPerLaunch = 256;
constexpr int kLookbackPerLane = 1;   // status words per lane per look-back round trip

// Status word: high 32 bits = (epoch tag << 2) | flag, low 32 bits = value.
constexpr unsigned kFlagInvalid = 0, kFlagAggregate = 1, kFlagInclusive = 2;

__device__ __forceinline__ unsigned long long pack_status(unsigned tag, unsigned flag, uint32_t bits)
{
    return (static_cast<unsigned long long>((tag << 2) | flag) << 32) | bits;
}

__device__ __forceinline__ unsigned long long ld_status(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_status(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Bit `nb` of the four words of v, gathered with byte permutes: byte nb / 8 of
// each word moves into one word (byte j from word j), whose bits nb % 8,
// 8 + nb % 8, ... then hold the four bits.  `sel` = byte_sel(nb), nbb = nb % 8.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint32_t byte_sel(int nb)
{
    const uint32_t b = static_cast<uint32_t>(nb) >> 3;
    return b | ((4u + b) << 4);
}
__device__ __forceinline__ uint32_t bytes_at_bit(const uint4 &v, uint32_t sel)
{
    const uint32_t lo = __byte_perm(v.x, v.y, sel), hi = __byte_perm(v.z, v.w, sel);
    return __byte_perm(lo, hi, 0x5410);
}
// how many of the four words have bit nb set
__device__ __forceinline__ uint32_t ones_at_bit(const uint4 &v, uint32_t sel, int nbb)
{
    return static_cast<uint32_t>(__popc((bytes_at_bit(v, sel) >> nbb) & 0x01010101u));
}
// bit j set when word j has bit nb set: the four bits at 0, 8, 16 and 24 land
// on bits 21 .. 24 of one product (1 + 2^7 + 2^14 + 2^21 has no two terms on
// one bit)
__device__ __forceinline__ uint32_t nibble_at_bit(const uint4 &v, uint32_t sel, int nbb)
{
    const uint32_t t = (bytes_at_bit(v, sel) >> nbb) & 0x01010101u;
    return ((t * 0x00204081u) >> 21) & 0xfu;
}

// ---------------------------------------------------------------------------
// Streaming global memory access (each element is read once and written once).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4 *p, uint4 v) { __stcs(p, v); }

// Load one tile row set.  `full`: the whole tile lies inside [0, n) and the
// pointer is 16-byte aligned, so every row is one 128-bit load.  Otherwise
// each element is loaded on its own, and elements past n read as `fill`.
template <typename S, int VECS, bool ALIGNED>
__device__ __forceinline__ void load_rows(const S *__restrict__ in, size_t warp_base, size_t n,
                                          int lane, bool full, S (&x)[VECS][4], S fill)
{
    if (ALIGNED && full) {
        uint4 q[VECS];
#pragma unroll
        for (int r = 0; r < VECS; ++r)
            q[r] = ld_stream(reinterpret_cast<const uint4 *>(in + warp_base) + r * 32 + lane);
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            x[r][0] = from_bits<S>(q[r].x);
            x[r][1] = from_bits<S>(q[r].y);
            x[r][2] = from_bits<S>(q[r].z);
            x[r][3] = from_bits<S>(q[r].w);
        }
    } else {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            size_t e = warp_base + static_cast<size_t>(r * 32 + lane) * 4;
            if (ALIGNED && e + 4 <= n) {
                uint4 q = ld_stream(reinterpret_cast<const uint4 *>(in + e));
                x[r][0] = from_bits<S>(q.x);
                x[r][1] = from_bits<S>(q.y);
                x[r][2] = from_bits<S>(q.z);
                x[r][3] = from_bits<S>(q.w);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) x[r][k] = (e + k < n) ? in[e + k] : fill;
            }
        }
    }
}

template <typename S, int VECS, bool ALIGNED>
__device__ __forceinline__ void store_rows(S *__restrict__ out, size_t warp_base, size_t n, int lane,
                                           bool full, const S (&y)[VECS][4])
{
    if (ALIGNED && full) {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            uint4 q = make_uint4(to_bits(y[r][0]), to_bits(y[r][1]), to_bits(y[r][2]), to_bits(y[r][3]));
            st_stream(reinterpret_cast<uint4 *>(out + warp_base) + r * 32 + lane, q);
        }
    } else {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            size_t e = warp_base + static_cast<size_t>(r * 32 + lane) * 4;
            if (ALIGNED && e + 4 <= n) {
                uint4 q = make_uint4(to_bits(y[r][0]), to_bits(y[r][1]), to_bits(y[r][2]), to_bits(y[r][3]));
                st_stream(reinterpret_cast<uint4 *>(out + e), q);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (e + k < n) out[e + k] = y[r][k];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Warp level: inclusive shuffle-up scan of each row's lane totals, all rows
// interleaved for instruction-level parallelism.  Lanes below `delta` have no
// source lane and keep their value (the guard the 5-step shuffle scan needs).
// Outputs, per row, the lane's exclusive prefix within the warp's run
// (earlier rows included) and the warp's total over all rows.
// ---------------------------------------------------------------------------
template <class Op, int VECS>
__device__ __forceinline__ void warp_scan_rows(const Op &op, const typename Op::S (&t)[VECS], int lane,
                                               typename Op::S (&excl)[VECS], typename Op::S &warp_total)
{
    using S = typename Op::S;
    S inc[VECS];
#pragma unroll
    for (int r = 0; r < VECS; ++r) inc[r] = t[r];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            S u = __shfl_up_sync(kFullMask, inc[r], d);
            if (lane >= d) inc[r] = op(u, inc[r]);
        }
    }
    S run = Op::identity();
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        S before = __shfl_up_sync(kFullMask, inc[r], 1);
        S row_total = __shfl_sync(kFullMask, inc[r], 31);
        excl[r] = (lane == 0) ? run : op(run, before);
        run = op(run, row_total);
    }
    warp_total = run;
}

// Block level: every warp scans the NWARPS warp totals held in shared memory
// and takes its own exclusive prefix and the tile total.
template <class Op, int NWARPS>
__device__ __forceinline__ void block_scan_warps(const Op &op, const typename Op::S *s_warp, int warp,
                                                 int lane, typename Op::S &warp_excl,
                                                 typename Op::S &tile_total)
{
    using S = typename Op::S;
    S v = (lane < NWARPS) ? s_warp[lane] : Op::identity();
#pragma unroll
    for (int d = 1; d < NWARPS; d <<= 1) {
        S u = __shfl_up_sync(kFullMask, v, d);
        if (lane >= d) v = op(u, v);
    }
    S before = __shfl_sync(kFullMask, v, (warp > 0) ? warp - 1 : 0);
    warp_excl = (warp > 0) ? before : Op::identity();
    tile_total = __shfl_sync(kFullMask, v, NWARPS - 1);
}

// ---------------------------------------------------------------------------
// Device level: decoupled look-back, run by one full warp.
//
// publish_aggregate: the tile's own total, flagged "aggregate" (tile 0
// publishes its total as "inclusive" straight away).
// lookback: the warp reads a window of predecessor status words.  It waits
// until every tile from the nearest predecessor down to the nearest
// "inclusive" one has published something, folds those values (aggregates
// plus the inclusive prefix), and either stops (an inclusive prefix was
// found) or moves the window further back.  Positions before tile 0 read as an
// inclusive identity.  Each wait is bounded by `spin_limit` polls; when it
// runs out the error word gets kErrTimeout and the result is not valid.
// ---------------------------------------------------------------------------
template <class Op>
__device__ __forceinline__ void publish(unsigned long long *status, unsigned tile, unsigned tag,
                                        unsigned flag, typename Op::S value, int lane)
{
    if (lane == 0) st_status(status + tile, pack_status(tag, flag, to_bits(value)));
}

// Look-back window: lane j reads the PER_LANE status words of tiles
// (end - 1 - PER_LANE * j - k), k = 0 .. PER_LANE - 1, so one round trip to
// L2 covers 32 * PER_LANE predecessors.  The rate at which tiles can finish
// is about (window size) / (L2 round-trip latency), so a wide window keeps
// the inter-block carry off the critical path.
template <class Op, int PER_LANE>
__device__ typename Op::S lookback(const Op &op, const unsigned long long *status, unsigned tile,
                                   unsigned tag, unsigned *error, unsigned spin_limit, int lane)
{
    using S = typename Op::S;
    S excl = Op::identity();
    long long end = static_cast<long long>(tile);
    bool gave_up = false;
    while (!gave_up) {
        unsigned flag[PER_LANE];
        uint32_t bits[PER_LANE];
        unsigned found;
        int upto;   // this lane's entries 0 .. upto contribute
        unsigned spins = 0;
        while (true) {
            unsigned long long w[PER_LANE];
#pragma unroll
            for (int k = 0; k < PER_LANE; ++k) {
                const long long idx = end - 1 - static_cast<long long>(PER_LANE) * lane - k;
                w[k] = (idx >= 0) ? ld_status(status + idx) : 0ull;
            }
            int kp = PER_LANE;   // this lane's nearest inclusive entry
#pragma unroll
            for (int k = PER_LANE - 1; k >= 0; --k) {
                const long long idx = end - 1 - static_cast<long long>(PER_LANE) * lane - k;
                if (idx >= 0) {
                    const unsigned hi = static_cast<unsigned>(w[k] >> 32);
                    flag[k] = ((hi >> 2) == tag) ? (hi & 3u) : kFlagInvalid;
                    bits[k] = static_cast<uint32_t>(w[k]);
                } else {
                    flag[k] = kFlagInclusive;
                    bits[k] = to_bits(Op::identity());
                }
                if (flag[k] == kFlagInclusive) kp = k;
            }
            found = __ballot_sync(kFullMask, kp < PER_LANE);
            const int jp = found ? __ffs(found) - 1 : 32;   // nearest lane holding an inclusive prefix
            upto = (lane < jp) ? PER_LANE - 1 : ((lane == jp) ? kp : -1);
            bool miss = false;
#pragma unroll
            for (int k = 0; k < PER_LANE; ++k) miss |= (k <= upto) && (flag[k] == kFlagInvalid);
            if (__ballot_sync(kFullMask, miss) == 0) break;
            if (++spins >= spin_limit) {
                if (lane == 0) atomicOr(error, kErrTimeout);
                gave_up = true;
                break;
            }
            if (spins > 4) __nanosleep(spins < 64 ? 32 : 256);
        }
        S v = Op::identity();
#pragma unroll
        for (int k = 0; k < PER_LANE; ++k)
            if (k <= upto && flag[k] != kFlagInvalid) v = op(from_bits<S>(bits[k]), v);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
        excl = op(v, excl);
        if (found) break;
        end -= 32LL * PER_LANE;
    }
    return excl;
}

// ---------------------------------------------------------------------------
// Two-level look-back.  Tiles form groups of 32.  Besides its own status
// word, the last tile of each group publishes a group status word: first
// the group's aggregate (the fold of its 32 tile aggregates, all of which
// its own level-1 window has seen), then the group's inclusive prefix.  A
// tile's look-back reads (1) the status words of its own group's earlier
// tiles -- at most 31, one round trip -- and, unless it met an inclusive
// prefix there, (2) the group status words of earlier groups, 32 groups
// (1,024 tiles) per round trip.  The inclusive frontier thus advances 1,024
// tiles per L2 round trip instead of 32.  Waits are bounded as above.
// Returns the tile's exclusive prefix; the caller publishes the tile's own
// status words, this function the group word.
// ---------------------------------------------------------------------------
// agg_inclusive: the tile's own status is already inclusive with value agg
// (a segmented scan's tile that contains a segment head): a group-closing
// tile then publishes agg itself as the group's inclusive word.
template <class Op>
__device__ typename Op::S lookback2(const Op &op, const unsigned long long *status,
                                    unsigned long long *status2, unsigned tile, unsigned tag,
                                    typename Op::S agg, unsigned *error, unsigned spin_limit, int lane,
                                    bool agg_inclusive = false)
{
    using S = typename Op::S;
    const unsigned group = tile >> 5;
    const long long first = static_cast<long long>(group) << 5;
    if (agg_inclusive && (tile & 31u) == 31u && lane == 0)
        st_status(status2 + group, pack_status(tag, kFlagInclusive, to_bits(agg)));
    const bool closes_group = !agg_inclusive && (tile & 31u) == 31u;
    bool gave_up = false;

    // level 1: this group's tiles first .. tile-1, lane j reading tile-1-j
    const long long idx = static_cast<long long>(tile) - 1 - lane;
    const bool mine = idx >= first;
    unsigned flag = kFlagInclusive, found, upto;
    uint32_t bits = to_bits(Op::identity());
    unsigned spins = 0;
    while (true) {
        if (mine) {
            const unsigned long long w = ld_status(status + idx);
            const unsigned hi = static_cast<unsigned>(w >> 32);
            flag = ((hi >> 2) == tag) ? (hi & 3u) : kFlagInvalid;
            bits = static_cast<uint32_t>(w);
        }
        found = __ballot_sync(kFullMask, mine && flag == kFlagInclusive);
        const unsigned in_group = __ballot_sync(kFullMask, mine);
        upto = found ? (((found & (0u - found)) << 1) - 1u) : in_group;
        const unsigned missing = __ballot_sync(kFullMask, mine && flag == kFlagInvalid);
        if ((missing & upto) == 0) break;
        if (++spins >= spin_limit) {
            if (lane == 0) atomicOr(error, kErrTimeout);
            gave_up = true;
            break;
        }
        if (spins > 4) __nanosleep(spins < 64 ? 32 : 256);
    }
    S v = (((upto >> lane) & 1u) && mine && flag != kFlagInvalid) ? from_bits<S>(bits) : Op::identity();
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
    const S level1 = v;   // fold of own-group predecessors back to an inclusive prefix, or all of them
    if (found || gave_up) {
        if (closes_group && lane == 0)
            st_status(status2 + group, pack_status(tag, kFlagInclusive, to_bits(op(level1, agg))));
        return level1;
    }
    if (closes_group && lane == 0)
        st_status(status2 + group, pack_status(tag, kFlagAggregate, to_bits(op(level1, agg))));

    // level 2: earlier groups, lane j reading group (end - 1 - j)
    S excl = Op::identity();
    long long end = static_cast<long long>(group);
    while (!gave_up) {
        const long long g = end - 1 - lane;
        unsigned gflag, gfound, gupto;
        uint32_t gbits;
        spins = 0;
        while (true) {
            if (g >= 0) {
                const unsigned long long w = ld_status(status2 + g);
                const unsigned hi = static_cast<unsigned>(w >> 32);
                gflag = ((hi >> 2) == tag) ? (hi & 3u) : kFlagInvalid;
                gbits = static_cast<uint32_t>(w);
            } else {
                gflag = kFlagInclusive;
                gbits = to_bits(Op::identity());
            }
            gfound = __ballot_sync(kFullMask, gflag == kFlagInclusive);
            gupto = gfound ? (((gfound & (0u - gfound)) << 1) - 1u) : kFullMask;
            const unsigned missing = __ballot_sync(kFullMask, gflag == kFlagInvalid);
            if ((missing & gupto) == 0) break;
            if (++spins >= spin_limit) {
                if (lane == 0) atomicOr(error, kErrTimeout);
                gave_up = true;
                break;
            }
            if (spins > 4) __nanosleep(spins < 64 ? 32 : 256);
        }
        S gv = (((gupto >> lane) & 1u) && gflag != kFlagInvalid) ? from_bits<S>(gbits) : Op::identity();
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) gv = op(gv, __shfl_xor_sync(kFullMask, gv, d));
        excl = op(gv, excl);
        if (gfound) break;
        end -= 32;
    }
    const S prefix = op(excl, level1);
    if (closes_group && lane == 0)
        st_status(status2 + group, pack_status(tag, kFlagInclusive, to_bits(op(prefix, agg))));
    return prefix;
}

// Run by lane 0 .. 31 of warp 0 of the block that owns the launch's last
// tile, after its look-back: every tile has published by then, so every
// block has read the epoch and taken its ticket.  Advances the epoch, resets
// the ticket counter and refreshes a rolling window of status slots that
// this launch did not use.
__device__ __forceinline__ void finish_launch(DevState *st, unsigned long long *status,
                                              unsigned num_tiles, unsigned capacity, int lane)
{
    __syncwarp();
    const unsigned cursor = st->cursor;
    if (capacity > num_tiles) {
        const unsigned spare = capacity - num_tiles;
        for (unsigned i = lane; i < kRefreshPerLaunch; i += 32)
            status[num_tiles + (cursor + i) % spare] = 0ull;
    }
    // group status words follow the tile status words (see group_status())
    unsigned long long *status2 = status + capacity;
    const unsigned groups = (num_tiles + 31u) >> 5, capacity2 = capacity >> 5;
    if (capacity2 > groups) {
        const unsigned spare = capacity2 - groups;
        for (unsigned i = lane; i < kRefreshPerLaunch; i += 32)
            status2[groups + (cursor + i) % spare] = 0ull;
    }
    __syncwarp();
    if (lane == 0) {
        st->cursor = cursor + kRefreshPerLaunch;
        st->ticket = 0u;
        const unsigned e = st->epoch + 1u;
        st->epoch = (e >= kEpochTags) ? 0u : e;
    }
}

// The group status words (capacity / 32 of them) sit right after the
// `capacity` tile status words in every workspace.
__device__ __forceinline__ unsigned long long *group_status(unsigned long long *status, unsigned capacity)
{
    return status + capacity;
}

__device__ __forceinline__ unsigned read_tag(const DevState *st)
{
    return *reinterpret_cast<const volatile unsigned *>(&st->epoch) + 1u;
}

}  // namespace devscan
