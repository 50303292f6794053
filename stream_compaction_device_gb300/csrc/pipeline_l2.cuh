// Persistent two-pass pipeline for sm_103a in which L2 holds each tile while
// its prefix is resolved.  One kernel template serves the scan, stream
// compaction and the one-bit split; a policy class P says what each pass
// loads and computes.
//
// Per tile t, in one block:
//   pass A     the A-producer warp takes tile tickets in order and
//              bulk-copies P's pass-A bytes of the tile into an A buffer
//              (L2 policy evict_last: pass B reads them again); the reduce
//              group folds them to the tile's aggregate (P::reduce), frees the
//              buffer, publishes the aggregate and only then claims one of R
//              in-flight tile records;
//   look-back  one warp per record runs the two-level decoupled look-back
//              (tile words plus group-of-32 words) for the tile's exclusive
//              prefix;
//   pass B     the B-producer warp, in record order, bulk-copies P's pass-B
//              bytes into a B buffer once the prefix is known (the bytes pass
//              A read are L2 hits); the consume group applies the prefix and
//              writes the output (P::consume).
// No block holds a tile's data while the look-back runs, so shared memory
// only has to cover load latency.  Every wait is bounded (the error word
// records a timeout); decisions after a group-wide wait are made uniform with
// a reducing barrier; both producers drain their bulk copies before the block
// exits.  The block that takes the launch's last ticket closes the launch
// (advances the epoch, resets the ticket counter).
#pragma once

#include "core.cuh"
#include "capture.cuh"
#include "grid_sync.cuh"
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

__device__ __forceinline__ uint64_t l2_policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 treatment of a bulk copy's lines.
enum L2Hint : int { kL2None = 0, kL2EvictLast = 1, kL2EvictFirst = 2, kL2EvictNormal = 3 };

__device__ __forceinline__ uint64_t l2_policy(int hint)
{
    return hint == kL2EvictLast ? l2_policy_evict_last()
                                : (hint == kL2EvictFirst ? l2_policy_evict_first() : l2_policy_evict_normal());
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

// Start moving `bytes` of global memory into L2 (no shared memory involved).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src_global, unsigned bytes, uint64_t policy)
{
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src_global), "r"(bytes),
                 "l"(policy)
                 : "memory");
}

// Named barrier ids of the pipeline (0 is __syncthreads).
constexpr unsigned kBarReduceDecide = 4, kBarReduceTotals = 5, kBarConsumeDecide = 6, kBarConsumeTotals = 7;

// Block-wide exclusive scan of the consume group's warp totals.  Every warp
// writes its total into buf[warp], the group meets at a named barrier, then
// each warp scans the NW totals.  Callers alternate between two buffers so a
// single barrier per call suffices.
template <class Op, int NW>
__device__ __forceinline__ void group_scan(const Op &op, typename Op::S warp_total, uint32_t *buf, int warp,
                                           int lane, typename Op::S &warp_excl, typename Op::S &group_total)
{
    using S = typename Op::S;
    if (lane == 0) buf[warp] = to_bits(warp_total);
    named_sync(kBarConsumeTotals, NW * 32);
    S v = (lane < NW) ? from_bits<S>(buf[lane]) : Op::identity();
#pragma unroll
    for (int d = 1; d < NW; d <<= 1) {
        const S u = __shfl_up_sync(kFullMask, v, d);
        if (lane >= d) v = op(u, v);
    }
    const S before = __shfl_sync(kFullMask, v, warp > 0 ? warp - 1 : 0);
    warp_excl = (warp > 0) ? before : Op::identity();
    group_total = __shfl_sync(kFullMask, v, NW - 1);
}

// A segmented policy (P::kSegmented) reports, per reduce warp, whether a
// segment head lies in the warp's contiguous part of the tile (`extra`
// nonzero) and folds only what follows the last head there; the kernel
// combines the warps in order, and a tile with a head publishes its
// aggregate as an inclusive prefix at once (nothing before the head can
// change it).
template <class P, class = void>
struct IsSegmented {
    static constexpr bool value = false;
};
template <class P>
struct IsSegmented<P, decltype(void(P::kSegmented))> {
    static constexpr bool value = P::kSegmented;
};

// Optional policy members, detected:
//   kParts        the reduce step also reports the aggregates of kParts equal
//                 parts of the tile (P::reduce_parts instead of P::reduce);
//                 the consume step gets their exclusive prefixes, so each
//                 consume warp knows its offset inside the tile without a
//                 group-wide scan.  Segmented policies report each part's
//                 value in part[q] and its head flag in part[kParts + q]; the
//                 tile's pair is their in-order fold, and the consume step
//                 gets the parts' own values with the head mask after them;
//   kScratchBytes shared memory for the consume group beyond the B buffers.
template <class P, class = void>
struct PolicyParts {
    static constexpr int value = 0;
};
template <class P>
struct PolicyParts<P, decltype(void(P::kParts))> {
    static constexpr int value = P::kParts;
};
//   kWarpIndependent  the consume step has no group-wide barrier: each
//                 consume warp waits for its B buffer on its own and may run
//                 ahead of the others by up to the ring's depth.
template <class P, class = void>
struct PolicyWarpIndependent {
    static constexpr bool value = false;
};
template <class P>
struct PolicyWarpIndependent<P, decltype(void(P::kWarpIndependent))> {
    static constexpr bool value = P::kWarpIndependent;
};
//   kAggregateAware  the policy sees each tile's aggregate: P::on_aggregate
//                 runs right after the reduce step publishes it, and pass B
//                 takes its copies from P::b_copies_for (given the
//                 aggregate) instead of P::b_copies.
template <class P, class = void>
struct PolicyAggregateAware {
    static constexpr bool value = false;
};
template <class P>
struct PolicyAggregateAware<P, decltype(void(P::kAggregateAware))> {
    static constexpr bool value = P::kAggregateAware;
};
//   kTicketBatch  tiles per ticket of the A producer (default 1): a ticket
//                 is one atomic on the stream's ticket counter, and the
//                 tiles of a ticket are consecutive and go to one block.
template <class P, class = void>
struct PolicyTicketBatch {
    static constexpr unsigned value = 1;
};
template <class P>
struct PolicyTicketBatch<P, decltype(void(P::kTicketBatch))> {
    static constexpr unsigned value = P::kTicketBatch;
};
// kCarryIn: tile 0's prefix is P::carry_prefix(args) -- the fold of
// whatever precedes the array (a shard's offset in a scan split across
// devices) -- and tile 0 publishes P::with_carry(args, aggregate) as its
// inclusive prefix.  Without a carry both leave the values as they were.
template <class P, class = void>
struct PolicyCarryIn {
    static constexpr bool value = false;
};
template <class P>
struct PolicyCarryIn<P, decltype(void(P::kCarryIn))> {
    static constexpr bool value = P::kCarryIn;
};

// A capturing policy (P::kCapturing) may do the whole job before the
// pipeline starts: when P::may_capture(args) (a cooperative launch), every
// block first runs P::capture over the whole of its dynamic shared memory
// and returns when it wrote the result; otherwise the pipeline starts from
// its usual state, which the capture does not touch.
template <class P, class = void>
struct PolicyCapturing {
    static constexpr bool value = false;
};
template <class P>
struct PolicyCapturing<P, decltype(void(P::kCapturing))> {
    static constexpr bool value = P::kCapturing;
};

template <class P, class = void>
struct PolicyScratch {
    static constexpr size_t value = 0;
};
template <class P>
struct PolicyScratch<P, decltype(void(P::kScratchBytes))> {
    static constexpr size_t value = P::kScratchBytes;
};

// Pass-A copies of tile t: P::a_copies when the policy has one (up to two
// copies, as for pass B), else the single copy P::a_src / P::a_bytes.
template <class P, class = void>
struct PassACopies {
    __device__ static void get(const typename P::Args &a, unsigned t, const void **src, unsigned *bytes,
                               unsigned *off)
    {
        src[0] = P::a_src(a, t);
        bytes[0] = P::a_bytes(a, t);
        off[0] = 0;
    }
};
template <class P>
struct PassACopies<P, decltype(void(&P::a_copies))> {
    __device__ static void get(const typename P::Args &a, unsigned t, const void **src, unsigned *bytes,
                               unsigned *off)
    {
        P::a_copies(a, t, src, bytes, off);
    }
};

// Finishes a reduce warp's part counts: c[i] is this lane's count of part
// rw + i * NR (each part's total is at most 2^15, so two parts share one
// word's 16-bit halves and one warp reduction); lane 0 stores the parts and
// returns their sum.
template <int PPW, int NR>
__device__ __forceinline__ unsigned store_part_counts(const unsigned (&c)[PPW], int rw, int lane, uint32_t *part)
{
    unsigned mine = 0;
#pragma unroll
    for (int i = 0; i < PPW; i += 2) {
        uint32_t w = c[i] | ((i + 1 < PPW) ? (c[i + 1] << 16) : 0u);
        w = __reduce_add_sync(kFullMask, w);
        if (lane == 0) {
            part[rw + i * NR] = w & 0xffffu;
            if (i + 1 < PPW) part[rw + (i + 1) * NR] = w >> 16;
        }
        mine += (w & 0xffffu) + (w >> 16);
    }
    return mine;
}

// What the consume group gets for one tile.
template <class S>
struct ConsumeTile {
    unsigned tile;
    S prefix;           // exclusive prefix of the tile's aggregate
    S aggregate;        // the tile's own aggregate (from pass A)
    unsigned char *buf; // the B buffer (P::kBBytes bytes)
    unsigned round;     // alternates the warp-totals buffers
    unsigned *warp_state;   // per-warp word kept across the block's tiles (0 at start)
    const uint32_t *part_excl;   // exclusive prefixes of the parts' aggregates (P::kParts > 0; until release;
                                 // segmented: the parts' values, then their head mask)
    unsigned char *scratch;      // P::kScratchBytes of shared memory for the consume group
};

template <class P>
struct PipeShape {
    static constexpr int NS = P::kConsumeWarps, NR = P::kReduceWarps, R = P::kRecords;
    static constexpr int SA = P::kAStages, SB = P::kBStages;
    static constexpr int kFirstReduceWarp = NS;
    static constexpr int kFirstLookbackWarp = NS + NR;
    static constexpr int kProducerA = NS + NR + R;
    static constexpr int kProducerB = NS + NR + R + 1;
    static constexpr int kThreads = (NS + NR + R + 2) * 32;
    static constexpr unsigned kNoCopy = 0xffffffffu;
    static constexpr int kParts = PolicyParts<P>::value;
    // segmented parts: the values, then one head flag per part (red_part) or
    // a mask of them (rec_part)
    static constexpr int kPartSlots = kParts > 0 ? (IsSegmented<P>::value ? 2 * kParts : kParts) : 1;
    struct Ctrl {
        uint64_t a_full[SA], a_empty[SA];
        uint64_t b_full[SB], b_empty[SB];
        uint64_t rec_pending[R], rec_ready[R], rec_free[R];
        unsigned a_tile[SA], a_last[SA];
        unsigned b_tile[SB], b_rec[SB], b_last[SB];
        unsigned rec_tile[R];
        uint32_t rec_agg[R], rec_prefix[R], rec_head[R];
        uint32_t red[NR], red_extra[NR];
        uint32_t red_part[kPartSlots], rec_part[R][kPartSlots];
        uint32_t wtot[2][NS];
        unsigned tag;
    };
    // Leading 16 bytes let a consume step read one chunk before B buffer 0.
    static constexpr size_t kLead = 16;
    static constexpr size_t kABase = kLead;
    static constexpr size_t kBBase = kABase + static_cast<size_t>(SA) * P::kABytes;
    static constexpr size_t kScratchBase = kBBase + static_cast<size_t>(SB) * P::kBBytes;
    static constexpr size_t kCtrlBase = kScratchBase + ((PolicyScratch<P>::value + 15) & ~static_cast<size_t>(15));
    static constexpr size_t kSmemBytes = kCtrlBase + sizeof(Ctrl) + 64;
    static_assert(P::kABytes % 16 == 0 && P::kBBytes % 16 == 0, "16-byte aligned buffers");
    static_assert(kThreads <= 1024, "one block of at most 1024 threads");
};

template <class P>
__global__ void __launch_bounds__(PipeShape<P>::kThreads, 1)
pipeline_l2_kernel(typename P::Args args, unsigned num_tiles, unsigned long long *status, DevState *st,
                   unsigned capacity, unsigned spin_limit, unsigned wait_limit)
{
    using Op = typename P::Op;
    using S = typename Op::S;
    using G = PipeShape<P>;
    constexpr int NS = G::NS, NR = G::NR, R = G::R, SA = G::SA, SB = G::SB;
    constexpr bool SEG = IsSegmented<P>::value;
    static_assert(!SEG || G::kParts > 0, "a segmented policy reports its parts' pairs");
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *abuf = smem + G::kABase;
    unsigned char *bbuf = smem + G::kBBase;
    auto *ctrl = reinterpret_cast<typename G::Ctrl *>(smem + G::kCtrlBase);
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // a capturing policy's back-off: nonzero when this call skips the capture
    // (its departure is counted by a look-back warp below, off the start)
    unsigned skipped_backoff = 0;
    if constexpr (PolicyCapturing<P>::value) {
        if (P::may_capture(args)) {
            const unsigned backoff = capture_backoff(st);
            if (backoff == 0u) {
                constexpr int NW = G::kThreads / 32;
                constexpr unsigned CAP = static_cast<unsigned>(G::kSmemBytes / 4 / NW);   // values per warp region
                if (P::template capture<NW, CAP>(args, reinterpret_cast<uint32_t *>(smem), st, spin_limit)) return;
                __syncthreads();   // every warp has left its region before the set-up below reuses the memory
            } else {
                skipped_backoff = backoff;
            }
        }
    }

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

    if (warp == G::kProducerA) {
        // ------------------------------------------------------- A producer
        // One ticket >= num_tiles per block ends the tickets; then R end
        // markers follow so that every look-back warp receives one.  With
        // D = P::kPrefetch > 0 the producer takes tickets D tiles ahead of
        // their A buffer and starts moving those tiles into L2 at once, so an
        // A buffer waits for an L2 hit rather than for HBM.  Lane j < D holds
        // the j-th queued ticket.
        constexpr int D = P::kPrefetch;
        static_assert(D >= 0 && D < 32, "prefetch depth");
        const uint64_t pol = l2_policy(P::kAHint);
        const uint64_t pre_pol = l2_policy_evict_last();
        bool tickets_done = false;
        // a ticket is a batch of K consecutive tiles (fewer atomic round
        // trips); a block still takes its tiles in order
        constexpr unsigned K = PolicyTicketBatch<P>::value;
        static_assert(K >= 1, "tiles per ticket");
        const unsigned batches = (num_tiles + K - 1) / K;
        unsigned batch_next = 0, batch_end = 0;   // tiles left of the current batch
        // takes the next tile (num_tiles once they are done) and, for a real
        // tile, starts its L2 prefetch
        auto take = [&]() -> unsigned {
            if (tickets_done) return num_tiles;
            if (batch_next >= batch_end) {
                unsigned b = 0;
                if (lane == 0) b = atomicAdd(&st->ticket, 1u);
                b = __shfl_sync(kFullMask, b, 0);
                if (b >= batches) {
                    tickets_done = true;
                    // the block that takes the launch's last ticket closes the launch
                    if (b == batches + gridDim.x - 1) finish_launch(st, status, num_tiles, capacity, lane);
                    return num_tiles;
                }
                batch_next = b * K;
                batch_end = batch_next + K < num_tiles ? batch_next + K : num_tiles;
            }
            const unsigned t = batch_next++;
            if (D > 0 && lane == 0) P::prefetch_l2(args, t, pre_pol);
            return t;
        };
        unsigned queued = num_tiles;
#pragma unroll 1
        for (int j = 0; j < D; ++j) {
            const unsigned t = take();
            if (lane == j) queued = t;
        }
        unsigned ends = 0;
        for (unsigned i = 0; ends < static_cast<unsigned>(R); ++i) {
            const unsigned a = i % SA, ka = i / SA;
            if (ka > 0 && !mbar_wait(&ctrl->a_empty[a], (ka - 1) & 1u, wait_limit)) {
                if (lane == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            unsigned t;
            if (D > 0) {
                t = __shfl_sync(kFullMask, queued, 0);
                queued = __shfl_down_sync(kFullMask, queued, 1);
            } else {
                t = take();
            }
            if (t >= num_tiles) {
                if (lane == 0) {
                    ctrl->a_tile[a] = num_tiles;
                    ctrl->a_last[a] = G::kNoCopy;
                    mbar_arrive(&ctrl->a_full[a]);
                }
                ++ends;
            } else if (lane == 0) {
                const void *src[2] = {nullptr, nullptr};
                unsigned bytes[2] = {0, 0}, off[2] = {0, 0};
                PassACopies<P>::get(args, t, src, bytes, off);
                const unsigned total = bytes[0] + bytes[1];
                ctrl->a_tile[a] = t;
                if (total != 0) {
                    ctrl->a_last[a] = ka;
                    mbar_arrive_expect_tx(&ctrl->a_full[a], total);
                    unsigned char *dst = abuf + static_cast<size_t>(a) * P::kABytes;
                    for (int j = 0; j < 2; ++j) {
                        if (bytes[j] == 0) continue;
                        if (P::kAHint == kL2None)
                            bulk_load(dst + off[j], src[j], bytes[j], &ctrl->a_full[a]);
                        else
                            bulk_load_hint(dst + off[j], src[j], bytes[j], &ctrl->a_full[a], pol);
                    }
                } else {
                    ctrl->a_last[a] = G::kNoCopy;
                    mbar_arrive(&ctrl->a_full[a]);
                }
            }
            // the next ticket only now: its atomic's round trip overlaps the
            // copy just issued instead of delaying it
            if (D > 0) {
                const unsigned nt = take();
                if (lane == D - 1) queued = nt;
            }
        }
        if (lane == 0)
            for (int a = 0; a < SA; ++a)
                if (ctrl->a_last[a] != G::kNoCopy) (void)mbar_wait(&ctrl->a_full[a], ctrl->a_last[a] & 1u, wait_limit);
        return;
    }

    if (warp == G::kProducerB) {
        // ------------------------------------------------------- B producer
        // Records in order (measured: serving them as their prefixes resolve
        // was slower -- the polling adds wake-up latency).
        const uint64_t pol = l2_policy(P::kBHint);
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
                ctrl->b_tile[b] = t < num_tiles ? t : num_tiles;
                ctrl->b_rec[b] = r;
                unsigned total = 0;
                const void *src[2] = {nullptr, nullptr};
                unsigned bytes[2] = {0, 0}, off[2] = {0, 0};
                if (t < num_tiles) {
                    if constexpr (PolicyAggregateAware<P>::value)
                        P::b_copies_for(args, t, from_bits<S>(ctrl->rec_agg[r]), src, bytes, off);
                    else
                        P::b_copies(args, t, src, bytes, off);
                    total = bytes[0] + bytes[1];
                }
                if (total != 0) {
                    ctrl->b_last[b] = kb;
                    mbar_arrive_expect_tx(&ctrl->b_full[b], total);
                    unsigned char *dst = bbuf + static_cast<size_t>(b) * P::kBBytes;
                    for (int j = 0; j < 2; ++j) {
                        if (bytes[j] == 0) continue;
                        if (P::kBHint == kL2None)
                            bulk_load(dst + off[j], src[j], bytes[j], &ctrl->b_full[b]);
                        else
                            bulk_load_hint(dst + off[j], src[j], bytes[j], &ctrl->b_full[b], pol);
                    }
                } else {
                    ctrl->b_last[b] = G::kNoCopy;
                    mbar_arrive(&ctrl->b_full[b]);
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
        if constexpr (PolicyCapturing<P>::value)
            if (skipped_backoff != 0u && r == 0 && lane == 0) capture_skip_depart(st, skipped_backoff, gridDim.x);
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
            const bool head = SEG && ctrl->rec_head[r] != 0;   // status already inclusive
            S prefix = Op::identity();
            if (t != 0) {
                prefix = lookback2<Op>(op, status, group_status(status, capacity), t, tag, agg, &st->error,
                                       spin_limit, lane, head);
                if (!head) publish<Op>(status, t, tag, kFlagInclusive, op(prefix, agg), lane);
            } else if constexpr (PolicyCarryIn<P>::value) {
                prefix = P::carry_prefix(args);
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
            if (!named_sync_and(kBarReduceDecide, NR * 32, landed)) {
                if (rtid == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
            const unsigned t = ctrl->a_tile[a];
            if (t >= num_tiles) {
                // forward the end marker to record r's look-back warp
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->a_empty[a]);
                bool freed = true;
                if (rtid == 0) {
                    if (kr > 0) freed = mbar_wait(&ctrl->rec_free[r], (kr - 1) & 1u, wait_limit);
                    if (!freed) atomicOr(&st->error, kErrTimeout);
                    ctrl->rec_tile[r] = num_tiles;
                    mbar_arrive(&ctrl->rec_pending[r]);
                }
                if (!named_sync_and(kBarReduceDecide, NR * 32, rtid != 0 || freed)) break;
                ++ends;
                continue;
            }
            S v = Op::identity();
            unsigned extra = 0;
            if constexpr (G::kParts > 0)
                P::reduce_parts(args, abuf + static_cast<size_t>(a) * P::kABytes, t, rtid, NR * 32, v, extra,
                                ctrl->red_part);
            else
                P::reduce(args, abuf + static_cast<size_t>(a) * P::kABytes, t, rtid, NR * 32, v, extra);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctrl->a_empty[a]);   // buffer read: free it
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
            if (P::kHasExtra) extra = __reduce_add_sync(kFullMask, extra);
            if (lane == 0) {
                ctrl->red[rw] = to_bits(v);
                ctrl->red_extra[rw] = extra;
            }
            named_sync(kBarReduceTotals, NR * 32);
            bool freed = true;
            if (rtid == 0) {
                S agg = from_bits<S>(ctrl->red[0]);
                unsigned ex = ctrl->red_extra[0];
                unsigned head = 0;
                // segmented parts: their values and head mask, read once
                uint32_t pval[SEG && G::kParts > 0 ? G::kParts : 1];
                unsigned pmask = 0;
                if constexpr (SEG && G::kParts > 0) {
#pragma unroll
                    for (int q = 0; q < G::kParts; ++q) {
                        pval[q] = ctrl->red_part[q];
                        if (ctrl->red_part[G::kParts + q] != 0) pmask |= 1u << q;
                    }
                    // in order: a part that holds a head restarts the fold
                    agg = Op::identity();
#pragma unroll
                    for (int q = 0; q < G::kParts; ++q)
                        agg = ((pmask >> q) & 1u) ? from_bits<S>(pval[q]) : op(agg, from_bits<S>(pval[q]));
                    head = pmask != 0 ? 1u : 0u;
                } else {
#pragma unroll
                    for (int w = 1; w < NR; ++w) {
                        agg = op(agg, from_bits<S>(ctrl->red[w]));
                        ex += ctrl->red_extra[w];
                    }
                }
                // publish first; a record (and so a look-back warp) is only
                // claimed for the time the prefix takes to resolve
                // tile 0 publishes its inclusive prefix: the carry-in (if
                // any) folded with its aggregate
                S pub = agg;
                if constexpr (PolicyCarryIn<P>::value)
                    if (t == 0) pub = P::with_carry(args, agg);
                st_status(status + t, pack_status(tag, (t == 0 || head) ? kFlagInclusive : kFlagAggregate,
                                                  to_bits(pub)));
                if (P::kHasExtra) P::after_reduce(args, t, ex);
                if constexpr (PolicyAggregateAware<P>::value) P::on_aggregate(args, t, agg);
                if (kr > 0) freed = mbar_wait(&ctrl->rec_free[r], (kr - 1) & 1u, wait_limit);
                if (!freed) atomicOr(&st->error, kErrTimeout);
                ctrl->rec_tile[r] = t;
                ctrl->rec_agg[r] = to_bits(agg);
                ctrl->rec_head[r] = head;
                if constexpr (SEG && G::kParts > 0) {
                    // the parts' own pairs: each consume warp combines those before it
#pragma unroll
                    for (int q = 0; q < G::kParts; ++q) ctrl->rec_part[r][q] = pval[q];
                    ctrl->rec_part[r][G::kParts] = pmask;
                } else if constexpr (G::kParts > 0) {
                    S acc = Op::identity();
                    for (int q = 0; q < G::kParts; ++q) {
                        ctrl->rec_part[r][q] = to_bits(acc);
                        acc = op(acc, from_bits<S>(ctrl->red_part[q]));
                    }
                }
                mbar_arrive(&ctrl->rec_pending[r]);
            }
            // red[] free for the next tile; a timed-out record wait ends the group
            if (!named_sync_and(kBarReduceTotals, NR * 32, rtid != 0 || freed)) break;
        }
        return;
    }

    // ----------------------------------------------------------- consume group
    unsigned round = 0;
    unsigned warp_state = 0;
    for (unsigned i = 0;; ++i) {
        const unsigned b = i % SB, kb = i / SB;
        const bool landed = mbar_wait(&ctrl->b_full[b], kb & 1u, wait_limit);
        if constexpr (PolicyWarpIndependent<P>::value) {
            // no barrier inside the consume step: a warp that gives up leaves
            // alone, and every wait of the others stays bounded
            if (!landed) {
                if (lane == 0) atomicOr(&st->error, kErrTimeout);
                break;
            }
        } else if (!named_sync_and(kBarConsumeDecide, NS * 32, landed)) {
            if (tid == 0) atomicOr(&st->error, kErrTimeout);
            break;
        }
        const unsigned t = ctrl->b_tile[b];
        if (t >= num_tiles) break;
        const unsigned r = ctrl->b_rec[b];
        ConsumeTile<S> ct;
        ct.tile = t;
        ct.prefix = from_bits<S>(ctrl->rec_prefix[r]);
        ct.aggregate = from_bits<S>(ctrl->rec_agg[r]);
        ct.buf = bbuf + static_cast<size_t>(b) * P::kBBytes;
        ct.round = round;
        ct.warp_state = &warp_state;
        ct.part_excl = ctrl->rec_part[r];
        ct.scratch = smem + G::kScratchBase;
        // release(): the B buffer and the record are no longer needed
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ctrl->b_empty[b]);
                mbar_arrive(&ctrl->rec_free[r]);
            }
        };
        round += P::consume(args, ct, ctrl->wtot[0], ctrl->wtot[1], warp, lane, release);
    }
}

// ---------------------------------------------------------------------------
// Scan policy: pass A reads the tile (4-byte elements) and folds it; pass B
// re-reads it, scans it with the prefix and stores it.
// ---------------------------------------------------------------------------
// AH / BH: L2 hints of the pass-A and pass-B copies; STREAM_OUT: evict-first
// (.cs) output stores.
// PARTS: pass A also folds each consume warp's 512-element part, so every
// consume warp starts from its own prefix and the consume step has no
// barrier; TB: tiles per ticket.
template <class OpT, bool INCLUSIVE, int NS_, int NR_, int VECS_, int SA_, int SB_, int R_, int AH = kL2EvictLast,
          int BH = kL2EvictFirst, bool STREAM_OUT = true, int PREFETCH = 0, bool PARTS = false, unsigned TB = 1>
struct ScanPolicy {
    using Op = OpT;
    static constexpr int kAHint = AH, kBHint = BH, kPrefetch = PREFETCH;
    using S = typename Op::S;
    static constexpr int kConsumeWarps = NS_, kReduceWarps = NR_, kRecords = R_, kAStages = SA_, kBStages = SB_;
    static constexpr int VECS = VECS_;
    static constexpr int kWarpItems = 32 * 4 * VECS;
    static constexpr int kTile = NS_ * 32 * 4 * VECS;
    static constexpr size_t kABytes = static_cast<size_t>(kTile) * 4;
    static constexpr size_t kBBytes = static_cast<size_t>(kTile) * 4;
    static constexpr bool kHasExtra = false;
    static constexpr int kParts = PARTS ? NS_ : 0;   // one part per consume warp
    static constexpr bool kWarpIndependent = PARTS;
    static constexpr unsigned kTicketBatch = TB;
    static constexpr bool kCarryIn = true;
    struct Args {
        const S *in;
        S *out;
        size_t n;
        const S *carry = nullptr;   // device word folded in front of the array, or null (identity)
    };
    __device__ static S carry_prefix(const Args &a) { return a.carry != nullptr ? *a.carry : Op::identity(); }
    __device__ static S with_carry(const Args &a, S v) { return a.carry != nullptr ? Op()(*a.carry, v) : v; }
    __device__ static unsigned tile_len(const Args &a, unsigned t)
    {
        const size_t rem = a.n - static_cast<size_t>(t) * kTile;
        return rem < static_cast<size_t>(kTile) ? static_cast<unsigned>(rem) : static_cast<unsigned>(kTile);
    }
    // elements a bulk copy delivers (a multiple of 16 bytes)
    __device__ static unsigned copied(const Args &a, unsigned t) { return tile_len(a, t) & ~3u; }
    __device__ static const void *a_src(const Args &a, unsigned t) { return a.in + static_cast<size_t>(t) * kTile; }
    __device__ static unsigned a_bytes(const Args &a, unsigned t) { return copied(a, t) * 4u; }
    __device__ static void prefetch_l2(const Args &a, unsigned t, uint64_t pol)
    {
        if (a_bytes(a, t) != 0) bulk_prefetch_l2(a_src(a, t), a_bytes(a, t), pol);
    }
    __device__ static void b_copies(const Args &a, unsigned t, const void **src, unsigned *bytes, unsigned *off)
    {
        src[0] = a.in + static_cast<size_t>(t) * kTile;
        bytes[0] = copied(a, t) * 4u;
        off[0] = 0;
    }
    __device__ static void reduce(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int nthr, S &v,
                                  unsigned &)
    {
        const Op op;
        const S *buf = reinterpret_cast<const S *>(abuf);
        const unsigned cp = copied(a, t);
        S v0 = Op::identity(), v1 = Op::identity(), v2 = Op::identity(), v3 = Op::identity();
        if (cp == static_cast<unsigned>(kTile)) {
            const uint4 *b4 = reinterpret_cast<const uint4 *>(buf);
#pragma unroll 4
            for (int c = rtid; c < kTile / 4; c += nthr) {
                const uint4 q = b4[c];
                v0 = op(v0, from_bits<S>(q.x));
                v1 = op(v1, from_bits<S>(q.y));
                v2 = op(v2, from_bits<S>(q.z));
                v3 = op(v3, from_bits<S>(q.w));
            }
        } else {
            const size_t base = static_cast<size_t>(t) * kTile;
            const unsigned len = tile_len(a, t);
            for (unsigned e = rtid; e < len; e += nthr) v0 = op(v0, e < cp ? buf[e] : a.in[base + e]);
        }
        v = op(op(v0, v1), op(v2, v3));
    }
    // pass A with parts: part q (consume warp q's kWarpItems elements) folded
    // into part[q]; reduce warp rw takes parts rw, rw + NR, ...; v: the fold
    // of this warp's parts in lane 0 (the kernel folds the lanes and warps)
    __device__ static void reduce_parts(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int, S &v,
                                        unsigned &, uint32_t *part)
    {
        static_assert(NS_ % NR_ == 0, "whole parts per reduce warp");
        constexpr int PPW = NS_ / NR_;
        const Op op;
        const int lane = rtid & 31, rw = rtid >> 5;
        const S *buf = reinterpret_cast<const S *>(abuf);
        const unsigned cp = copied(a, t), len = tile_len(a, t);
        const size_t base = static_cast<size_t>(t) * kTile;
        // every part's loads first, then the folds and stores: a store to
        // part[] between them would keep the next part's loads behind it
        S pv[PPW];
        if (cp == static_cast<unsigned>(kTile)) {
#pragma unroll
            for (int i = 0; i < PPW; ++i) {
                const uint4 *b4 = reinterpret_cast<const uint4 *>(buf + (rw + i * NR_) * kWarpItems);
                pv[i] = Op::identity();
#pragma unroll
                for (int k = 0; k < VECS; ++k) {
                    const uint4 u = b4[k * 32 + lane];
                    pv[i] = op(pv[i], op(op(from_bits<S>(u.x), from_bits<S>(u.y)), op(from_bits<S>(u.z), from_bits<S>(u.w))));
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < PPW; ++i) {
                const unsigned p0 = static_cast<unsigned>((rw + i * NR_) * kWarpItems);
                pv[i] = Op::identity();
                for (unsigned e = p0 + lane; e < p0 + kWarpItems && e < len; e += 32)
                    pv[i] = op(pv[i], e < cp ? buf[e] : a.in[base + e]);
            }
        }
        S mine = Op::identity();
#pragma unroll
        for (int i = 0; i < PPW; ++i) {
            const S w = warp_fold(op, pv[i]);
            if (lane == 0) part[rw + i * NR_] = to_bits(w);
            mine = op(mine, w);
        }
        v = (lane == 0) ? mine : Op::identity();
    }
    __device__ static void after_reduce(const Args &, unsigned, unsigned) {}
    // This warp's rows of the consumed tile, from the B buffer (elements past
    // the bulk copy from global memory; past n the identity).
    __device__ static void load_x(const Args &a, const ConsumeTile<S> &ct, int warp, int lane, S (&x)[VECS][4])
    {
        const unsigned t = ct.tile;
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        const S *buf = reinterpret_cast<const S *>(ct.buf);
        const unsigned cp = copied(a, t);
        if (cp == static_cast<unsigned>(kTile)) {
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
                    x[q][j] = (e < cp) ? buf[e] : ((base + e < a.n) ? a.in[base + e] : Op::identity());
                }
        }
    }
    // Scans the rows in place (inclusive or exclusive, the tile's prefix
    // applied); returns the tile's own total.  Contains the consume group's
    // barrier.
    __device__ static S scan_x(const ConsumeTile<S> &ct, uint32_t *wbuf0, uint32_t *wbuf1, int warp, int lane,
                               S (&x)[VECS][4])
    {
        const Op op;
        S tt[VECS];
#pragma unroll
        for (int q = 0; q < VECS; ++q) tt[q] = op(op(x[q][0], x[q][1]), op(x[q][2], x[q][3]));
        S row_excl[VECS], warp_total;
        warp_scan_rows<Op, VECS>(op, tt, lane, row_excl, warp_total);
        S warp_excl, total;
        group_scan<Op, NS_>(op, warp_total, (ct.round & 1) ? wbuf1 : wbuf0, warp, lane, warp_excl, total);
        const S pfx = op(ct.prefix, warp_excl);
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
        return total;
    }
    __device__ static void store_x(S *out, size_t n, unsigned t, int warp, int lane, const S (&x)[VECS][4])
    {
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        if (base + kTile <= n) {
            uint4 *o4 = reinterpret_cast<uint4 *>(out + base + wbase);
#pragma unroll
            for (int q = 0; q < VECS; ++q) {
                const uint4 v = make_uint4(to_bits(x[q][0]), to_bits(x[q][1]), to_bits(x[q][2]), to_bits(x[q][3]));
                if (STREAM_OUT)
                    st_stream(o4 + q * 32 + lane, v);
                else
                    o4[q * 32 + lane] = v;
            }
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
    // Scans the rows in place from `pfx`, the prefix of this warp's part
    // (no barrier: the parts' prefixes come from pass A).
    __device__ static void scan_x_from(S pfx, int lane, S (&x)[VECS][4])
    {
        const Op op;
        S tt[VECS];
#pragma unroll
        for (int q = 0; q < VECS; ++q) tt[q] = op(op(x[q][0], x[q][1]), op(x[q][2], x[q][3]));
        S row_excl[VECS], warp_total;
        warp_scan_rows<Op, VECS>(op, tt, lane, row_excl, warp_total);
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
    }
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *wbuf0, uint32_t *wbuf1,
                                       int warp, int lane, Release &release)
    {
        S x[VECS][4];
        load_x(a, ct, warp, lane, x);
        if constexpr (PARTS) {
            const Op op;
            const S pfx = op(ct.prefix, from_bits<S>(ct.part_excl[warp]));
            release();   // the tile and the part's prefix are in registers now
            scan_x_from(pfx, lane, x);
            store_x(a.out, a.n, ct.tile, warp, lane, x);
            return 0;
        } else {
            release();   // the tile is in registers now
            scan_x(ct, wbuf0, wbuf1, warp, lane, x);
            store_x(a.out, a.n, ct.tile, warp, lane, x);
            return 1;   // one warp-totals buffer used
        }
    }
};

}  // namespace devscan
