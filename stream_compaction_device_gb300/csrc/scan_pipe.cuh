// Persistent, warp-specialised single-pass scan for sm_103a.
//
// Each block owns a ring of STAGES tile buffers in shared memory and runs
// four roles at once:
//   producer warp    takes tile tickets in order and fills free buffers with
//                    1-D bulk (TMA) copies from global memory;
//   local-scan group NA warps: as soon as a tile lands they scan it inside
//                    the block (thread-serial, shuffle-up warp scan, block
//                    scan over warp totals), write the tile-local scan back
//                    into the buffer and publish the tile aggregate;
//   look-back warps  one per buffer: the decoupled two-level look-back for
//                    the tile's exclusive prefix;
//   store group      NB warps, tiles in order: combine the prefix into the
//                    tile-local scan and write it out with 128-bit stores,
//                    then free the buffer.
// A tile's aggregate is therefore published about one local scan after its
// data arrives, and the look-back latency overlaps with the loads and local
// scans of the tiles behind it; the buffers (not registers) hold the data
// while the prefix is resolved.
//
// Requirements: `in` and `out` 16-byte aligned (the host falls back to the
// one-tile-per-block kernel otherwise).  All waits are bounded; a wait that
// runs out sets the error word, decisions after a timeout are made uniform
// across a group with a reducing barrier, and the producer drains its
// outstanding bulk copies before the block exits.
#pragma once

#include "core.cuh"
#include "pipeline.cuh"

namespace devscan {

// NA local-scan warps, NB store warps, VECS 16-byte rows per local-scan
// thread and sub-tile, SUB sub-tiles per tile, STAGES buffers (= look-back
// warps).
template <int NA, int NB, int VECS, int SUB, int STAGES>
struct PipeGeom {
    static constexpr int kScanThreads = NA * 32;
    static constexpr int kStoreThreads = NB * 32;
    static constexpr int kFirstStoreWarp = NA;
    static constexpr int kFirstLookbackWarp = NA + NB;
    static constexpr int kProducerWarp = NA + NB + STAGES;
    static constexpr int kThreads = (NA + NB + STAGES + 1) * 32;
    static constexpr int kWarpItems = 32 * 4 * VECS;
    static constexpr int kSubTile = kScanThreads * 4 * VECS;
    static constexpr int kTile = kSubTile * SUB;
    static constexpr size_t kStageBytes = static_cast<size_t>(kTile) * 4;
    static constexpr unsigned kNoCopy = 0xffffffffu;
    struct Ctrl {
        uint64_t full[STAGES];     // producer arrive + bulk-copy bytes
        uint64_t scanned[STAGES];  // one arrival per local-scan warp
        uint64_t ready[STAGES];    // look-back warp: prefix known
        uint64_t empty[STAGES];    // one arrival per store warp: buffer free
        unsigned tile[STAGES];
        unsigned copied[STAGES];   // elements delivered by the bulk copy
        uint32_t agg[STAGES];      // tile aggregate (bits)
        uint32_t prefix[STAGES];   // tile exclusive prefix (bits)
        unsigned last_copy_phase[STAGES];
        uint32_t wtot[2][NA];
        unsigned tag;
    };
    static constexpr size_t kSmemBytes = STAGES * kStageBytes + sizeof(Ctrl);
};

// Named barrier ids (0 is __syncthreads).
constexpr unsigned kBarScanDecide = 1, kBarScanTotals = 2, kBarStoreDecide = 3;

template <class Op, bool INCLUSIVE, int NA, int NB, int VECS, int SUB, int STAGES>
__global__ void __launch_bounds__((NA + NB + STAGES + 1) * 32, 1)
scan_pipe_kernel(const typename Op::S *__restrict__ in, typename Op::S *__restrict__ out, size_t n,
                 unsigned num_tiles, unsigned long long *status, DevState *st, unsigned capacity,
                 unsigned spin_limit, unsigned wait_limit)
{
    using S = typename Op::S;
    using G = PipeGeom<NA, NB, VECS, SUB, STAGES>;
    constexpr int TILE = G::kTile;
    extern __shared__ __align__(128) unsigned char smem[];
    S *stages = reinterpret_cast<S *>(smem);
    auto *ctrl = reinterpret_cast<typename G::Ctrl *>(smem + STAGES * G::kStageBytes);
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&ctrl->full[s], 1);
            mbar_init(&ctrl->scanned[s], NA);
            mbar_init(&ctrl->ready[s], 1);
            mbar_init(&ctrl->empty[s], NB);
            ctrl->last_copy_phase[s] = G::kNoCopy;
        }
        ctrl->tag = read_tag(st);
        mbar_init_fence();
    }
    __syncthreads();
    const unsigned tag = ctrl->tag;

    if (warp == G::kProducerWarp) {
        // ------------------------------------------------------------ producer
        // Tickets run out with one ticket >= num_tiles per block; after it the
        // producer puts an end marker into every buffer so that each
        // look-back warp (one per buffer) sees one.
        unsigned ends = 0;
        for (unsigned i = 0; ends < static_cast<unsigned>(STAGES); ++i) {
            const unsigned s = i % STAGES, k = i / STAGES;
            if (k > 0 && !mbar_wait(&ctrl->empty[s], (k - 1) & 1u, wait_limit)) {
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
                    ctrl->tile[s] = num_tiles;
                    ctrl->last_copy_phase[s] = G::kNoCopy;
                    mbar_arrive(&ctrl->full[s]);
                }
                // the block that takes the launch's last ticket closes the launch
                if (ends == 0 && t == num_tiles + gridDim.x - 1) finish_launch(st, status, num_tiles, capacity, lane);
                ++ends;
                continue;
            }
            if (lane == 0) {
                const size_t base = static_cast<size_t>(t) * TILE;
                const size_t rem = n - base;
                const unsigned len = rem < static_cast<size_t>(TILE) ? static_cast<unsigned>(rem) : TILE;
                const unsigned bytes = (len * static_cast<unsigned>(sizeof(S))) & ~15u;
                ctrl->tile[s] = t;
                ctrl->copied[s] = bytes / static_cast<unsigned>(sizeof(S));
                if (bytes != 0) {
                    ctrl->last_copy_phase[s] = k;
                    mbar_arrive_expect_tx(&ctrl->full[s], bytes);
                    bulk_load(stages + static_cast<size_t>(s) * TILE, in + base, bytes, &ctrl->full[s]);
                } else {
                    ctrl->last_copy_phase[s] = G::kNoCopy;
                    mbar_arrive(&ctrl->full[s]);
                }
            }
        }
        // no bulk copy may still be writing this block's shared memory when it exits
        if (lane == 0)
            for (int s = 0; s < STAGES; ++s)
                if (ctrl->last_copy_phase[s] != G::kNoCopy)
                    (void)mbar_wait(&ctrl->full[s], ctrl->last_copy_phase[s] & 1u, wait_limit);
        return;
    }

    if (warp >= G::kFirstLookbackWarp) {
        // --------------------------------------------------- look-back warp s
        const unsigned s = static_cast<unsigned>(warp - G::kFirstLookbackWarp);
        for (unsigned k = 0;; ++k) {
            if (!mbar_wait(&ctrl->full[s], k & 1u, wait_limit)) {
                if (lane == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            const unsigned t = ctrl->tile[s];
            if (t >= num_tiles) {
                if (lane == 0) mbar_arrive(&ctrl->ready[s]);
                break;
            }
            if (!mbar_wait(&ctrl->scanned[s], k & 1u, wait_limit)) {
                if (lane == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            const S agg = from_bits<S>(ctrl->agg[s]);
            S prefix = Op::identity();
            if (t != 0) {
                prefix = lookback2<Op>(op, status, group_status(status, capacity), t, tag, agg, &st->error,
                                       spin_limit, lane);
                publish<Op>(status, t, tag, kFlagInclusive, op(prefix, agg), lane);
            }
            if (lane == 0) {
                ctrl->prefix[s] = to_bits(prefix);
                mbar_arrive(&ctrl->ready[s]);
            }
        }
        return;
    }

    if (warp < NA) {
        // ----------------------------------------------------- local-scan group
        unsigned round = 0;   // selects the warp-totals buffer
        for (unsigned i = 0;; ++i) {
            const unsigned s = i % STAGES, k = i / STAGES;
            const bool landed = mbar_wait(&ctrl->full[s], k & 1u, wait_limit);
            if (!named_sync_and(kBarScanDecide, G::kScanThreads, landed)) {
                if (tid == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            const unsigned t = ctrl->tile[s];
            if (t >= num_tiles) break;
            const unsigned copied = ctrl->copied[s];
            const size_t base = static_cast<size_t>(t) * TILE;
            S *buf = stages + static_cast<size_t>(s) * TILE;
            S carry = Op::identity();
#pragma unroll 1
            for (int sub = 0; sub < SUB; ++sub, ++round) {
                const int wbase = sub * G::kSubTile + warp * G::kWarpItems;
                S x[VECS][4];
                if (copied == static_cast<unsigned>(TILE)) {
                    const uint4 *b4 = reinterpret_cast<const uint4 *>(buf + wbase);
#pragma unroll
                    for (int r = 0; r < VECS; ++r) {
                        const uint4 q = b4[r * 32 + lane];
                        x[r][0] = from_bits<S>(q.x);
                        x[r][1] = from_bits<S>(q.y);
                        x[r][2] = from_bits<S>(q.z);
                        x[r][3] = from_bits<S>(q.w);
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < VECS; ++r)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const unsigned e = static_cast<unsigned>(wbase + (r * 32 + lane) * 4 + j);
                            x[r][j] = (e < copied) ? buf[e] : ((base + e < n) ? in[base + e] : Op::identity());
                        }
                }
                S tt[VECS];
#pragma unroll
                for (int r = 0; r < VECS; ++r) tt[r] = op(op(x[r][0], x[r][1]), op(x[r][2], x[r][3]));
                S row_excl[VECS], warp_total;
                warp_scan_rows<Op, VECS>(op, tt, lane, row_excl, warp_total);
                if (lane == 0) ctrl->wtot[round & 1][warp] = to_bits(warp_total);
                named_sync(kBarScanTotals, G::kScanThreads);
                S wv = (lane < NA) ? from_bits<S>(ctrl->wtot[round & 1][lane]) : Op::identity();
#pragma unroll
                for (int d = 1; d < NA; d <<= 1) {
                    const S u = __shfl_up_sync(kFullMask, wv, d);
                    if (lane >= d) wv = op(u, wv);
                }
                const S before = __shfl_sync(kFullMask, wv, warp > 0 ? warp - 1 : 0);
                const S sub_total = __shfl_sync(kFullMask, wv, NA - 1);
                const S pfx = (warp > 0) ? op(carry, before) : carry;
#pragma unroll
                for (int r = 0; r < VECS; ++r) {
                    S cur = op(pfx, row_excl[r]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
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
                // the tile-local scan goes back into the buffer
                uint4 *w4 = reinterpret_cast<uint4 *>(buf + wbase);
#pragma unroll
                for (int r = 0; r < VECS; ++r)
                    w4[r * 32 + lane] =
                        make_uint4(to_bits(x[r][0]), to_bits(x[r][1]), to_bits(x[r][2]), to_bits(x[r][3]));
                carry = op(carry, sub_total);
            }
            if (tid == 0) {
                ctrl->agg[s] = to_bits(carry);
                // tile 0's aggregate is its inclusive prefix
                st_status(status + t, pack_status(tag, t == 0 ? kFlagInclusive : kFlagAggregate, to_bits(carry)));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->scanned[s]);
        }
        return;
    }

    // ------------------------------------------------------------ store group
    const int sw = warp - G::kFirstStoreWarp;
    for (unsigned i = 0;; ++i) {
        const unsigned s = i % STAGES, k = i / STAGES;
        const bool ready = mbar_wait(&ctrl->ready[s], k & 1u, wait_limit);
        if (!named_sync_and(kBarStoreDecide, G::kStoreThreads, ready)) {
            if (sw == 0 && lane == 0) atomicOr(&st->error, kErrTimeout);
            break;
        }
        const unsigned t = ctrl->tile[s];
        if (t >= num_tiles) break;
        const S prefix = from_bits<S>(ctrl->prefix[s]);
        const size_t base = static_cast<size_t>(t) * TILE;
        const S *buf = stages + static_cast<size_t>(s) * TILE;
        const uint4 *b4 = reinterpret_cast<const uint4 *>(buf);
        uint4 *o4 = reinterpret_cast<uint4 *>(out + base);
        const int c0 = sw * 32 + lane;
        if (base + TILE <= n) {
#pragma unroll 4
            for (int c = c0; c < TILE / 4; c += G::kStoreThreads) {
                const uint4 q = b4[c];
                st_stream(o4 + c,
                          make_uint4(to_bits(op(prefix, from_bits<S>(q.x))), to_bits(op(prefix, from_bits<S>(q.y))),
                                     to_bits(op(prefix, from_bits<S>(q.z))), to_bits(op(prefix, from_bits<S>(q.w)))));
            }
        } else {
            for (int c = c0; c < TILE / 4; c += G::kStoreThreads)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const size_t e = base + 4u * c + j;
                    if (e < n) out[e] = op(prefix, buf[4 * c + j]);
                }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctrl->empty[s]);
    }
}

}  // namespace devscan
