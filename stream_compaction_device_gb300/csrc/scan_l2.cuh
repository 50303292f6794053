// Persistent single-pass scan for sm_103a that lets L2 hold each tile while
// its prefix is resolved.
//
// Per tile, in one block:
//   pass A  the A-producer warp bulk-copies the tile from HBM into an A
//           buffer (L2 policy evict_last); the reduce group folds it to the
//           tile aggregate, frees the buffer, publishes the aggregate and
//           only then claims an in-flight tile record -- the data is not
//           held in the block while the look-back runs;
//   look-back  one warp per in-flight tile record runs the two-level
//           decoupled look-back and records the tile's exclusive prefix;
//   pass B  the B-producer warp, in tile order, bulk-copies the tile again
//           into a B buffer (an L2 hit; policy evict_first) once its prefix
//           is known; the scan group scans it (thread-serial, shuffle-up warp
//           scan, block scan over warp totals), combines the prefix and
//           writes the result with 128-bit stores.
// HBM traffic stays at one read and one write per element as long as the
// tile is still in L2 when pass B re-reads it (the look-back takes a few
// microseconds; L2 holds far more than the bytes read in that time).
//
// Requirements: `in` and `out` 16-byte aligned; n a multiple of 4 elements
// or the last tile's remainder is read with ordinary loads.  Every wait is
// bounded; group decisions after a wait are made uniform with a reducing
// barrier; both producers drain their bulk copies before the block exits.
#pragma once

#include "core.cuh"
#include "pipeline.cuh"

namespace devscan {

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_load_hint(void *dst_smem, const void *src_global, unsigned bytes, uint64_t *bar,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst_smem)),
        "l"(src_global), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// NS scan warps (VECS rows each), NR reduce warps, SA / SB buffers, R
// records (= look-back warps).
template <int NS, int NR, int VECS, int SA, int SB, int R>
struct L2Geom {
    static constexpr int kScanThreads = NS * 32;
    static constexpr int kReduceThreads = NR * 32;
    static constexpr int kFirstReduceWarp = NS;
    static constexpr int kFirstLookbackWarp = NS + NR;
    static constexpr int kProducerA = NS + NR + R;
    static constexpr int kProducerB = NS + NR + R + 1;
    static constexpr int kThreads = (NS + NR + R + 2) * 32;
    static constexpr int kWarpItems = 32 * 4 * VECS;
    static constexpr int kTile = kScanThreads * 4 * VECS;
    static constexpr size_t kStageBytes = static_cast<size_t>(kTile) * 4;
    static constexpr unsigned kNoCopy = 0xffffffffu;
    struct Ctrl {
        uint64_t a_full[SA], a_empty[SA];
        uint64_t b_full[SB], b_empty[SB];
        uint64_t rec_pending[R], rec_ready[R], rec_free[R];
        unsigned a_tile[SA], a_copied[SA], a_last[SA];
        unsigned b_tile[SB], b_copied[SB], b_last[SB];
        unsigned rec_tile[R];
        uint32_t rec_agg[R], rec_prefix[R];
        uint32_t red[NR];
        uint32_t wtot[2][NS];
        unsigned tag;
    };
    static constexpr size_t kSmemBytes = (SA + SB) * kStageBytes + sizeof(Ctrl);
};

constexpr unsigned kBarReduceDecide = 4, kBarReduceTotals = 5, kBarL2ScanDecide = 6, kBarL2ScanTotals = 7;

template <class Op, bool INCLUSIVE, int NS, int NR, int VECS, int SA, int SB, int R>
__global__ void __launch_bounds__((NS + NR + R + 2) * 32, 1)
scan_l2_kernel(const typename Op::S *__restrict__ in, typename Op::S *__restrict__ out, size_t n,
               unsigned num_tiles, unsigned long long *status, DevState *st, unsigned capacity,
               unsigned spin_limit, unsigned wait_limit)
{
    using S = typename Op::S;
    using G = L2Geom<NS, NR, VECS, SA, SB, R>;
    constexpr int TILE = G::kTile;
    extern __shared__ __align__(128) unsigned char smem[];
    S *abuf = reinterpret_cast<S *>(smem);
    S *bbuf = abuf + static_cast<size_t>(SA) * TILE;
    auto *ctrl = reinterpret_cast<typename G::Ctrl *>(smem + (SA + SB) * G::kStageBytes);
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(&ctrl->a_full[s], 1);
            mbar_init(&ctrl->a_empty[s], NR);
            ctrl->a_last[s] = G::kNoCopy;
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(&ctrl->b_full[s], 1);
            mbar_init(&ctrl->b_empty[s], NS);
            ctrl->b_last[s] = G::kNoCopy;
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(&ctrl->rec_pending[r], 1);
            mbar_init(&ctrl->rec_ready[r], 1);
            mbar_init(&ctrl->rec_free[r], NS);
        }
        ctrl->tag = read_tag(st);
        mbar_init_fence();
    }
    __syncthreads();
    const unsigned tag = ctrl->tag;

    // element count a bulk copy can deliver for tile t (a multiple of 16 bytes)
    auto copy_elems = [&](unsigned t) -> unsigned {
        const size_t base = static_cast<size_t>(t) * TILE;
        const size_t rem = n - base;
        const unsigned len = rem < static_cast<size_t>(TILE) ? static_cast<unsigned>(rem) : TILE;
        return ((len * static_cast<unsigned>(sizeof(S))) & ~15u) / static_cast<unsigned>(sizeof(S));
    };

    if (warp == G::kProducerA) {
        // ------------------------------------------------------- A producer
        // One ticket >= num_tiles per block ends the tickets; then R end
        // markers follow so that every look-back warp receives one.
        const uint64_t pol = l2_policy_evict_last();
        unsigned ends = 0;
        for (unsigned i = 0; ends < static_cast<unsigned>(R); ++i) {
            const unsigned a = i % SA, ka = i / SA;
            const bool ok = (ka == 0) || mbar_wait(&ctrl->a_empty[a], (ka - 1) & 1u, wait_limit);
            if (!ok) {
                if (lane == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            unsigned t = num_tiles;
            if (ends == 0) {
                if (lane == 0) t = atomicAdd(&st->ticket, 1u);
                t = __shfl_sync(kFullMask, t, 0);
            }
            if (t >= num_tiles) {
                if (lane == 0) {
                    ctrl->a_tile[a] = num_tiles;
                    ctrl->a_last[a] = G::kNoCopy;
                    mbar_arrive(&ctrl->a_full[a]);
                }
                if (ends == 0 && t == num_tiles + gridDim.x - 1) finish_launch(st, status, num_tiles, capacity, lane);
                ++ends;
                continue;
            }
            if (lane == 0) {
                const unsigned elems = copy_elems(t);
                ctrl->a_tile[a] = t;
                ctrl->a_copied[a] = elems;
                if (elems != 0) {
                    ctrl->a_last[a] = ka;
                    mbar_arrive_expect_tx(&ctrl->a_full[a], elems * static_cast<unsigned>(sizeof(S)));
                    bulk_load_hint(abuf + static_cast<size_t>(a) * TILE, in + static_cast<size_t>(t) * TILE,
                                   elems * static_cast<unsigned>(sizeof(S)), &ctrl->a_full[a], pol);
                } else {
                    ctrl->a_last[a] = G::kNoCopy;
                    mbar_arrive(&ctrl->a_full[a]);
                }
            }
        }
        if (lane == 0)
            for (int a = 0; a < SA; ++a)
                if (ctrl->a_last[a] != G::kNoCopy) (void)mbar_wait(&ctrl->a_full[a], ctrl->a_last[a] & 1u, wait_limit);
        return;
    }

    if (warp == G::kProducerB) {
        // ------------------------------------------------------- B producer
        const uint64_t pol = l2_policy_evict_first();
        for (unsigned i = 0;; ++i) {
            const unsigned b = i % SB, kb = i / SB, r = i % R, kr = i / R;
            bool ok = mbar_wait(&ctrl->rec_ready[r], kr & 1u, wait_limit);
            if (ok && kb > 0) ok = mbar_wait(&ctrl->b_empty[b], (kb - 1) & 1u, wait_limit);
            if (!ok) {
                if (lane == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            const unsigned t = ctrl->rec_tile[r];
            if (lane == 0) {
                if (t >= num_tiles) {
                    ctrl->b_tile[b] = num_tiles;
                    ctrl->b_last[b] = G::kNoCopy;
                    mbar_arrive(&ctrl->b_full[b]);
                } else {
                    const unsigned elems = copy_elems(t);
                    ctrl->b_tile[b] = t;
                    ctrl->b_copied[b] = elems;
                    if (elems != 0) {
                        ctrl->b_last[b] = kb;
                        mbar_arrive_expect_tx(&ctrl->b_full[b], elems * static_cast<unsigned>(sizeof(S)));
                        bulk_load_hint(bbuf + static_cast<size_t>(b) * TILE, in + static_cast<size_t>(t) * TILE,
                                       elems * static_cast<unsigned>(sizeof(S)), &ctrl->b_full[b], pol);
                    } else {
                        ctrl->b_last[b] = G::kNoCopy;
                        mbar_arrive(&ctrl->b_full[b]);
                    }
                }
            }
            if (t >= num_tiles) break;
        }
        if (lane == 0)
            for (int b = 0; b < SB; ++b)
                if (ctrl->b_last[b] != G::kNoCopy) (void)mbar_wait(&ctrl->b_full[b], ctrl->b_last[b] & 1u, wait_limit);
        return;
    }

    if (warp >= G::kFirstLookbackWarp) {
        // ------------------------------------------------ look-back warp r
        const unsigned r = static_cast<unsigned>(warp - G::kFirstLookbackWarp);
        for (unsigned k = 0;; ++k) {
            if (!mbar_wait(&ctrl->rec_pending[r], k & 1u, wait_limit)) {
                if (lane == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            const unsigned t = ctrl->rec_tile[r];
            if (t >= num_tiles) {
                if (lane == 0) mbar_arrive(&ctrl->rec_ready[r]);
                break;
            }
            const S agg = from_bits<S>(ctrl->rec_agg[r]);
            S prefix = Op::identity();
            if (t != 0) {
                prefix = lookback2<Op>(op, status, group_status(status, capacity), t, tag, agg, &st->error,
                                       spin_limit, lane);
                publish<Op>(status, t, tag, kFlagInclusive, op(prefix, agg), lane);
            }
            if (lane == 0) {
                ctrl->rec_prefix[r] = to_bits(prefix);
                mbar_arrive(&ctrl->rec_ready[r]);
            }
        }
        return;
    }

    if (warp >= G::kFirstReduceWarp) {
        // ---------------------------------------------------- reduce group
        const int rw = warp - G::kFirstReduceWarp;
        const int rtid = rw * 32 + lane;
        unsigned ends = 0;
        for (unsigned i = 0; ends < static_cast<unsigned>(R); ++i) {
            const unsigned a = i % SA, ka = i / SA, r = i % R, kr = i / R;
            const bool landed = mbar_wait(&ctrl->a_full[a], ka & 1u, wait_limit);
            if (!named_sync_and(kBarReduceDecide, G::kReduceThreads, landed)) {
                if (rtid == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            const unsigned t = ctrl->a_tile[a];
            if (t >= num_tiles) {
                // forward the end marker to record r's look-back warp
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->a_empty[a]);
                bool freed = true;
                if (rtid == 0 && kr > 0) freed = mbar_wait(&ctrl->rec_free[r], (kr - 1) & 1u, wait_limit);
                if (rtid == 0) {
                    if (!freed) atomicOr(&st->error, kErrTimeout);
                    ctrl->rec_tile[r] = num_tiles;
                    mbar_arrive(&ctrl->rec_pending[r]);
                }
                if (!named_sync_and(kBarReduceDecide, G::kReduceThreads, rtid != 0 || freed)) break;
                ++ends;
                continue;
            }
            const unsigned copied = ctrl->a_copied[a];
            const size_t base = static_cast<size_t>(t) * TILE;
            const S *buf = abuf + static_cast<size_t>(a) * TILE;
            S v0 = Op::identity(), v1 = Op::identity(), v2 = Op::identity(), v3 = Op::identity();
            if (copied == static_cast<unsigned>(TILE)) {
                const uint4 *b4 = reinterpret_cast<const uint4 *>(buf);
#pragma unroll 4
                for (int c = rtid; c < TILE / 4; c += G::kReduceThreads) {
                    const uint4 q = b4[c];
                    v0 = op(v0, from_bits<S>(q.x));
                    v1 = op(v1, from_bits<S>(q.y));
                    v2 = op(v2, from_bits<S>(q.z));
                    v3 = op(v3, from_bits<S>(q.w));
                }
            } else {
                for (int c = rtid; c < TILE / 4; c += G::kReduceThreads)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const unsigned e = 4u * c + j;
                        if (e < copied)
                            v0 = op(v0, buf[e]);
                        else if (base + e < n)
                            v0 = op(v0, in[base + e]);
                    }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->a_empty[a]);   // buffer read: free it
            S v = op(op(v0, v1), op(v2, v3));
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
            if (lane == 0) ctrl->red[rw] = to_bits(v);
            named_sync(kBarReduceTotals, G::kReduceThreads);
            bool freed = true;
            if (rtid == 0) {
                S agg = from_bits<S>(ctrl->red[0]);
#pragma unroll
                for (int w = 1; w < NR; ++w) agg = op(agg, from_bits<S>(ctrl->red[w]));
                // publish first; a record (and so a look-back warp) is only
                // claimed for the time the prefix takes to resolve
                st_status(status + t, pack_status(tag, t == 0 ? kFlagInclusive : kFlagAggregate, to_bits(agg)));
                if (kr > 0) freed = mbar_wait(&ctrl->rec_free[r], (kr - 1) & 1u, wait_limit);
                if (!freed) atomicOr(&st->error, kErrTimeout);
                ctrl->rec_tile[r] = t;
                ctrl->rec_agg[r] = to_bits(agg);
                mbar_arrive(&ctrl->rec_pending[r]);
            }
            // red[] free for the next tile; a timed-out record wait ends the group
            if (!named_sync_and(kBarReduceTotals, G::kReduceThreads, rtid != 0 || freed)) break;
        }
        return;
    }

    // ---------------------------------------------------------- scan group
    unsigned round = 0;
    for (unsigned i = 0;; ++i, ++round) {
        const unsigned b = i % SB, kb = i / SB, r = i % R;
        const bool landed = mbar_wait(&ctrl->b_full[b], kb & 1u, wait_limit);
        if (!named_sync_and(kBarL2ScanDecide, G::kScanThreads, landed)) {
            if (tid == 0) atomicOr(&st->error, kErrTimeout);
            break;
        }
        const unsigned t = ctrl->b_tile[b];
        if (t >= num_tiles) break;
        const unsigned copied = ctrl->b_copied[b];
        const S prefix = from_bits<S>(ctrl->rec_prefix[r]);
        const size_t base = static_cast<size_t>(t) * TILE;
        const int wbase = warp * G::kWarpItems;
        const S *buf = bbuf + static_cast<size_t>(b) * TILE;
        S x[VECS][4];
        if (copied == static_cast<unsigned>(TILE)) {
            const uint4 *b4 = reinterpret_cast<const uint4 *>(buf + wbase);
#pragma unroll
            for (int q = 0; q < VECS; ++q) {
                const uint4 u = b4[q * 32 + lane];
                x[q][0] = from_bits<S>(u.x);
                x[q][1] = from_bits<S>(u.y);
                x[q][2] = from_bits<S>(u.z);
                x[q][3] = from_bits<S>(u.w);
            }
        } else {
#pragma unroll
            for (int q = 0; q < VECS; ++q)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const unsigned e = static_cast<unsigned>(wbase + (q * 32 + lane) * 4 + j);
                    x[q][j] = (e < copied) ? buf[e] : ((base + e < n) ? in[base + e] : Op::identity());
                }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&ctrl->b_empty[b]);
            mbar_arrive(&ctrl->rec_free[r]);
        }
        S tt[VECS];
#pragma unroll
        for (int q = 0; q < VECS; ++q) tt[q] = op(op(x[q][0], x[q][1]), op(x[q][2], x[q][3]));
        S row_excl[VECS], warp_total;
        warp_scan_rows<Op, VECS>(op, tt, lane, row_excl, warp_total);
        if (lane == 0) ctrl->wtot[round & 1][warp] = to_bits(warp_total);
        named_sync(kBarL2ScanTotals, G::kScanThreads);
        S wv = (lane < NS) ? from_bits<S>(ctrl->wtot[round & 1][lane]) : Op::identity();
#pragma unroll
        for (int d = 1; d < NS; d <<= 1) {
            const S u = __shfl_up_sync(kFullMask, wv, d);
            if (lane >= d) wv = op(u, wv);
        }
        const S before = __shfl_sync(kFullMask, wv, warp > 0 ? warp - 1 : 0);
        const S pfx = (warp > 0) ? op(prefix, before) : prefix;
#pragma unroll
        for (int q = 0; q < VECS; ++q) {
            S cur = op(pfx, row_excl[q]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const S v = x[q][j];
                if (INCLUSIVE) {
                    cur = op(cur, v);
                    x[q][j] = cur;
                } else {
                    x[q][j] = cur;
                    cur = op(cur, v);
                }
            }
        }
        if (base + TILE <= n) {
            uint4 *o4 = reinterpret_cast<uint4 *>(out + base + wbase);
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
                    if (e < n) out[e] = x[q][j];
                }
        }
    }
}

}  // namespace devscan
