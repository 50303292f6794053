// Device-wide inclusive / exclusive scan kernels (sm_103a).
//
// Inter-block carry strategies (geek-doc.cn "并行前缀和 scan ..." section 四
// describes the three-phase one and mentions chaining blocks in one launch):
//   * pipelined single pass (default for 16-byte-aligned data): persistent
//     warp-specialised blocks; bulk copies, tile aggregates published as
//     soon as a tile lands, two-level decoupled look-back, and L2 holding
//     each tile while its prefix resolves (pipeline_l2.cuh); one launch, HBM
//     traffic about 2 * n * sizeof(T) bytes;
//   * one tile per block with decoupled look-back (any 4-byte alignment):
//     one launch, 2 * n * sizeof(T) bytes, but each block holds its tile in
//     registers for the whole look-back;
//   * reduce-then-scan: tile totals, one-block scan of the totals, then the
//     tile scan with its offset -- three launches and one extra read of the
//     input (3 * n * sizeof(T) bytes).
#include "core.cuh"
#include "launch.h"
#include "scan_kernel.cuh"
#include "pipeline_l2.cuh"

#include <atomic>

namespace devscan {

// ---------------------------------------------------------------------------
// Reduce-then-scan: (1) tile totals, (2) exclusive scan of the totals in one
// block, (3) tile scan seeded with the tile's offset.
// ---------------------------------------------------------------------------
template <class Op, int THREADS, int VECS, bool ALIGNED>
__global__ void __launch_bounds__(THREADS)
rts_reduce_kernel(const typename Op::S *__restrict__ in, size_t n, typename Op::S *__restrict__ tile_sums)
{
    using S = typename Op::S;
    constexpr int NWARPS = THREADS / 32;
    constexpr int WARP_ITEMS = 32 * 4 * VECS;
    constexpr int TILE = THREADS * 4 * VECS;
    __shared__ S s_warp[NWARPS];
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned tile = blockIdx.x;
    const size_t tile_base = static_cast<size_t>(tile) * TILE;
    const size_t warp_base = tile_base + static_cast<size_t>(warp) * WARP_ITEMS;
    const bool full = tile_base + TILE <= n;
    S x[VECS][4];
    load_rows<S, VECS, ALIGNED>(in, warp_base, n, lane, full, x, Op::identity());
    S v = Op::identity();
#pragma unroll
    for (int r = 0; r < VECS; ++r) v = op(v, op(op(x[r][0], x[r][1]), op(x[r][2], x[r][3])));
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
    if (lane == 0) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        S w = (lane < NWARPS) ? s_warp[lane] : Op::identity();
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) w = op(w, __shfl_xor_sync(kFullMask, w, d));
        if (lane == 0) tile_sums[tile] = w;
    }
}

// One block of 1024 threads scans `count` tile totals in place (exclusive),
// 4 per thread per round, carrying the running total between rounds.
template <class Op>
__global__ void __launch_bounds__(1024) rts_scan_sums_kernel(typename Op::S *sums, unsigned count)
{
    using S = typename Op::S;
    constexpr int NWARPS = 32;
    __shared__ S s_warp[NWARPS];
    __shared__ S s_carry;
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_carry = Op::identity();
    __syncthreads();
    for (unsigned base = 0; base < count; base += 4096) {
        S x[1][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const unsigned i = base + tid * 4 + k;
            x[0][k] = (i < count) ? sums[i] : Op::identity();
        }
        S t[1] = {op(op(x[0][0], x[0][1]), op(x[0][2], x[0][3]))};
        S row_excl[1], warp_total;
        warp_scan_rows<Op, 1>(op, t, lane, row_excl, warp_total);
        if (lane == 0) s_warp[warp] = warp_total;
        __syncthreads();
        S warp_excl, block_total;
        block_scan_warps<Op, NWARPS>(op, s_warp, warp, lane, warp_excl, block_total);
        const S carry = s_carry;
        S cur = op(op(carry, warp_excl), row_excl[0]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const unsigned i = base + tid * 4 + k;
            const S v = x[0][k];
            if (i < count) sums[i] = cur;
            cur = op(cur, v);
        }
        __syncthreads();
        if (tid == 0) s_carry = op(carry, block_total);
        __syncthreads();
    }
}

template <class Op, int THREADS, int VECS, bool INCLUSIVE, bool ALIGNED>
__global__ void __launch_bounds__(THREADS)
rts_downsweep_kernel(const typename Op::S *__restrict__ in, typename Op::S *__restrict__ out, size_t n,
                     const typename Op::S *__restrict__ tile_prefix)
{
    using S = typename Op::S;
    constexpr int NWARPS = THREADS / 32;
    constexpr int WARP_ITEMS = 32 * 4 * VECS;
    constexpr int TILE = THREADS * 4 * VECS;
    __shared__ S s_warp[NWARPS];
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned tile = blockIdx.x;
    const size_t tile_base = static_cast<size_t>(tile) * TILE;
    const size_t warp_base = tile_base + static_cast<size_t>(warp) * WARP_ITEMS;
    const bool full = tile_base + TILE <= n;
    S x[VECS][4];
    load_rows<S, VECS, ALIGNED>(in, warp_base, n, lane, full, x, Op::identity());
    S t[VECS];
#pragma unroll
    for (int r = 0; r < VECS; ++r) t[r] = op(op(x[r][0], x[r][1]), op(x[r][2], x[r][3]));
    S row_excl[VECS], warp_total;
    warp_scan_rows<Op, VECS>(op, t, lane, row_excl, warp_total);
    if (lane == 0) s_warp[warp] = warp_total;
    __syncthreads();
    S warp_excl, tile_total;
    block_scan_warps<Op, NWARPS>(op, s_warp, warp, lane, warp_excl, tile_total);
    const S pfx = op(tile_prefix[tile], warp_excl);
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
    store_rows<S, VECS, ALIGNED>(out, warp_base, n, lane, full, x);
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait: one warp looks back from tile 1 onto a
// status slot that nothing ever publishes (its word is zero, which no epoch
// tag matches), gives up after `spin_limit` polls and records the timeout.
// ---------------------------------------------------------------------------
__global__ void stalled_wait_kernel(const unsigned long long *never_published, DevState *st,
                                    unsigned spin_limit)
{
    const AddU32 op;
    const unsigned tag = read_tag(st);
    (void)lookback<AddU32, kLookbackPerLane>(op, never_published, 1u, tag, &st->error, spin_limit, threadIdx.x & 31);
}

// ---------------------------------------------------------------------------
// Host-side launchers.
// ---------------------------------------------------------------------------
namespace {

template <class Op, bool INCLUSIVE, bool ALIGNED>
cudaError_t launch_lookback(const void *in, void *out, size_t n, const Workspace &ws, unsigned spin_limit,
                            cudaStream_t s, const void *carry_in)
{
    using S = typename Op::S;
    constexpr int THREADS = kScanThreads, VECS = kScanVecs;
    const unsigned tiles = tiles_for(n, kScanTile);
    scan_lookback_kernel<Op, THREADS, VECS, INCLUSIVE, ALIGNED, kUseTickets><<<tiles, THREADS, 0, s>>>(
        static_cast<const S *>(in), static_cast<S *>(out), n, tiles, ws.status, ws.state, ws.capacity,
        spin_limit, NoEpilogue::Args{}, static_cast<const S *>(carry_in));
    return cudaGetLastError();
}

// Geometry of the pipelined scan: 16 consume warps x 4 rows (8,192-element
// tiles), 4 reduce warps, 2 A buffers, 4 B buffers, 10 in-flight records
// (1,024 threads, about 193 KiB of shared memory: one block per SM); tiles
// are taken one ahead and prefetched into L2.  Chosen by sweeps on GB300:
// the reduce step sits on the A ring's turnaround, so four reduce warps beat
// two (by 3-4%); deeper prefetch and more records overflow what L2 keeps.
// Pass A also folds each consume warp's part, so the consume warps need no
// barrier, and a ticket hands out two tiles: together 1.2% faster at 2^28
// (either alone gained nothing, two tiles per ticket alone lost 3%).
constexpr unsigned kWaitLimit = 1u << 18;   // bounded mbarrier polls (~1 us each at most)
constexpr size_t kPipelineMinN = size_t(1) << 20;
// Sizes the L2-resident scan takes by default: measured on GB300 (L2 flushed
// between calls) it beats the one-tile kernel from 2^17 and the pipeline up
// to 2^24 by 10-40%, and loses above, once the input no longer stays in L2
// between its two reads.
constexpr size_t kL2ResidentMinN = size_t(1) << 17, kL2ResidentMaxN = size_t(1) << 24;

template <class Op, bool INCLUSIVE>
cudaError_t launch_pipelined(const void *in, void *out, size_t n, const Workspace &ws, unsigned spin_limit,
                             cudaStream_t s, const void *carry_in)
{
    using S = typename Op::S;
    using P = ScanPolicy<Op, INCLUSIVE, 16, 4, 4, 2, 4, 10, kL2EvictLast, kL2EvictFirst, true, 1, true, 2>;
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
    typename P::Args args{static_cast<const S *>(in), static_cast<S *>(out), n, static_cast<const S *>(carry_in)};
    kernel<<<grid, G::kThreads, G::kSmemBytes, s>>>(args, tiles, ws.status, ws.state, ws.capacity, spin_limit,
                                                    kWaitLimit);
    return cudaGetLastError();
}

template <class Op, bool INCLUSIVE>
cudaError_t launch_rts(const void *in, void *out, size_t n, const Workspace &ws, cudaStream_t s)
{
    using S = typename Op::S;
    constexpr int THREADS = kScanThreads, VECS = kScanVecs;
    const unsigned tiles = tiles_for(n, kScanTile);
    S *sums = reinterpret_cast<S *>(ws.tile_sums);
    rts_reduce_kernel<Op, THREADS, VECS, true><<<tiles, THREADS, 0, s>>>(static_cast<const S *>(in), n, sums);
    rts_scan_sums_kernel<Op><<<1, 1024, 0, s>>>(sums, tiles);
    rts_downsweep_kernel<Op, THREADS, VECS, INCLUSIVE, true><<<tiles, THREADS, 0, s>>>(
        static_cast<const S *>(in), static_cast<S *>(out), n, sums);
    return cudaGetLastError();
}

template <class Op, bool INCLUSIVE>
cudaError_t dispatch_op(const void *in, void *out, size_t n, bool aligned, int carry, const Workspace &ws,
                        unsigned spin_limit, cudaStream_t s, const void *carry_in)
{
    // reduce-then-scan has no carry-in: a scan with one takes the look-back
    if (carry == kCarryReduceThenScan && aligned && carry_in == nullptr) return launch_rts<Op, INCLUSIVE>(in, out, n, ws, s);
    // up to 2^19 elements the pipeline's fill latency outweighs its
    // bandwidth: one tile per block is faster there (measured on GB300)
    const bool pipelined = aligned && (carry == kCarryPipelined || (carry == kCarryDefault && n >= kPipelineMinN));
    if (pipelined) return launch_pipelined<Op, INCLUSIVE>(in, out, n, ws, spin_limit, s, carry_in);
    if (aligned) return launch_lookback<Op, INCLUSIVE, true>(in, out, n, ws, spin_limit, s, carry_in);
    return launch_lookback<Op, INCLUSIVE, false>(in, out, n, ws, spin_limit, s, carry_in);
}

template <class Op>
cudaError_t dispatch_dir(const void *in, void *out, size_t n, bool inclusive, bool aligned, int carry,
                         const Workspace &ws, unsigned spin_limit, cudaStream_t s, const void *carry_in)
{
    return inclusive ? dispatch_op<Op, true>(in, out, n, aligned, carry, ws, spin_limit, s, carry_in)
                     : dispatch_op<Op, false>(in, out, n, aligned, carry, ws, spin_limit, s, carry_in);
}

}  // namespace

cudaError_t launch_scan(ElemType type, int op, bool inclusive, const void *in, void *out, size_t n,
                        bool aligned, int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s,
                        const void *carry_in)
{
    // small inputs: one thread-block cluster (scan_cluster.cu)
    if (carry == kCarryDefault && n <= kClusterMaxN)
        return launch_scan_cluster(type, op, inclusive, in, out, n, aligned, s, carry_in);
    // inputs that fit in L2: one cooperative launch (scan_l2res.cu)
    if (aligned && (carry == kCarryL2Resident ||
                    (carry == kCarryDefault && n >= kL2ResidentMinN && n <= kL2ResidentMaxN)))
        return launch_scan_l2_resident(type, op, inclusive, in, out, n, ws, spin_limit, s, carry_in);
    switch (type) {
    case ElemType::I32:
        if (op == kOpAdd) return dispatch_dir<AddU32>(in, out, n, inclusive, aligned, carry, ws, spin_limit, s, carry_in);
        if (op == kOpMax) return dispatch_dir<MaxI32>(in, out, n, inclusive, aligned, carry, ws, spin_limit, s, carry_in);
        return dispatch_dir<XorU32>(in, out, n, inclusive, aligned, carry, ws, spin_limit, s, carry_in);
    case ElemType::U32:
        if (op == kOpAdd) return dispatch_dir<AddU32>(in, out, n, inclusive, aligned, carry, ws, spin_limit, s, carry_in);
        if (op == kOpMax) return dispatch_dir<MaxU32>(in, out, n, inclusive, aligned, carry, ws, spin_limit, s, carry_in);
        return dispatch_dir<XorU32>(in, out, n, inclusive, aligned, carry, ws, spin_limit, s, carry_in);
    case ElemType::F32:
        if (op == kOpAdd) return dispatch_dir<AddF32>(in, out, n, inclusive, aligned, carry, ws, spin_limit, s, carry_in);
        return dispatch_dir<MaxF32>(in, out, n, inclusive, aligned, carry, ws, spin_limit, s, carry_in);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_stalled_wait(const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    stalled_wait_kernel<<<1, 32, 0, s>>>(ws.never_published, ws.state, spin_limit);
    return cudaGetLastError();
}

}  // namespace devscan
