// Single-pass look-back scan kernel template (sm_103a), shared by the
// translation units that instantiate it.
#pragma once

#include "core.cuh"

namespace devscan {

// Work a scan kernel may do on each finished tile besides storing it.
struct NoEpilogue {
    struct Args {};
    static constexpr bool kActive = false;
    template <class S, int VECS>
    __device__ static void tile(const Args &, const S (&)[VECS][4], bool, S, int, int)
    {
    }
};

// ---------------------------------------------------------------------------
// Single-pass scan: one tile per block.
// ---------------------------------------------------------------------------
// LB: status words per lane of a look-back round trip; MINB: resident blocks
// per SM the register allocation must allow; EPI: per-tile epilogue (it sees
// the scanned rows, whether the tile is the last one, and the tile's
// inclusive prefix).  With an active epilogue a null `out` skips the store.
// carry_in: a device word that seeds tile 0's prefix (the fold of whatever
// precedes the array), or null for the identity.
template <class Op, int THREADS, int VECS, bool INCLUSIVE, bool ALIGNED, bool TICKETS,
          int LB = kLookbackPerLane, int MINB = 1, bool TWO_LEVEL = false, class EPI = NoEpilogue>
__global__ void __launch_bounds__(THREADS, MINB)
scan_lookback_kernel(const typename Op::S *__restrict__ in, typename Op::S *__restrict__ out, size_t n,
                     unsigned num_tiles, unsigned long long *status, DevState *st, unsigned capacity,
                     unsigned spin_limit, typename EPI::Args epi = typename EPI::Args{},
                     const typename Op::S *carry_in = nullptr)
{
    using S = typename Op::S;
    constexpr int NWARPS = THREADS / 32;
    constexpr int WARP_ITEMS = 32 * 4 * VECS;
    constexpr int TILE = THREADS * 4 * VECS;
    __shared__ S s_warp[NWARPS];
    __shared__ S s_prefix;
    __shared__ unsigned s_tile;
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    unsigned tile;
    if (TICKETS) {
        if (tid == 0) s_tile = atomicAdd(&st->ticket, 1u);
        __syncthreads();
        tile = s_tile;
        if (tile >= num_tiles) return;   // never taken: each launch hands out exactly num_tiles tickets
    } else {
        tile = blockIdx.x;
    }
    const size_t tile_base = static_cast<size_t>(tile) * TILE;
    const size_t warp_base = tile_base + static_cast<size_t>(warp) * WARP_ITEMS;
    const bool full = tile_base + TILE <= n;

    S x[VECS][4];
    load_rows<S, VECS, ALIGNED>(in, warp_base, n, lane, full, x, Op::identity());

    // thread level: serial combine of the 4 elements of each row
    S t[VECS];
#pragma unroll
    for (int r = 0; r < VECS; ++r) t[r] = op(op(x[r][0], x[r][1]), op(x[r][2], x[r][3]));

    S row_excl[VECS], warp_total;
    warp_scan_rows<Op, VECS>(op, t, lane, row_excl, warp_total);
    if (lane == 0) s_warp[warp] = warp_total;
    __syncthreads();

    S warp_excl, tile_total;
    block_scan_warps<Op, NWARPS>(op, s_warp, warp, lane, warp_excl, tile_total);

    if (warp == 0) {
        const unsigned tag = __shfl_sync(kFullMask, lane == 0 ? read_tag(st) : 0u, 0);
        S prefix = Op::identity();
        if (tile == 0) {
            if (carry_in != nullptr) prefix = *carry_in;
            publish<Op>(status, tile, tag, kFlagInclusive, carry_in != nullptr ? op(prefix, tile_total) : tile_total,
                        lane);
        } else {
            publish<Op>(status, tile, tag, kFlagAggregate, tile_total, lane);
            if (TWO_LEVEL)
                prefix = lookback2<Op>(op, status, group_status(status, capacity), tile, tag, tile_total,
                                       &st->error, spin_limit, lane);
            else
                prefix = lookback<Op, LB>(op, status, tile, tag, &st->error, spin_limit, lane);
            publish<Op>(status, tile, tag, kFlagInclusive, op(prefix, tile_total), lane);
        }
        if (lane == 0) s_prefix = prefix;
        if (tile == num_tiles - 1) finish_launch(st, status, num_tiles, capacity, lane);
    }
    __syncthreads();

    const S pfx = op(s_prefix, warp_excl);
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        S cur = op(pfx, row_excl[r]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const S v = x[r][k];
            if (INCLUSIVE) {
                cur = op(cur, v);
                x[r][k] = cur;
            } else {
                x[r][k] = cur;
                cur = op(cur, v);
            }
        }
    }
    if (EPI::kActive) {
        EPI::template tile<S, VECS>(epi, x, tile == num_tiles - 1, op(s_prefix, tile_total), tid, lane);
        if (out == nullptr) return;
    }
    store_rows<S, VECS, ALIGNED>(out, warp_base, n, lane, full, x);
}

}  // namespace devscan
