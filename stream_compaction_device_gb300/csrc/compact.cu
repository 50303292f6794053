// Stream compaction, fused into one single-pass kernel (sm_103a).
//
// geek-doc.cn "并行前缀和 scan ..." section 一 and lpnh.cn "并行扫描" section
// 4.1: each kept element's output slot is the exclusive add-scan of the 0/1
// predicate; pgsm.cn "SIMT数据依赖与并行前缀和" section 4.2: the two-kernel
// block-count variant and the last thread writing the total.  Here the
// predicate scan, the inter-block carry (decoupled look-back on kept
// counts), the staged scatter and the count all happen in one launch that
// reads values and flags once and writes only the kept values.
#include <atomic>

#include "core.cuh"
#include "launch.h"
#include "compact_policy.cuh"
#include "pipeline_l2.cuh"
#include "stage.cuh"

namespace devscan {

// GT: keep in[i] when (int32) in[i] > threshold (flags unused); otherwise
// keep it when flags[i] != 0.
template <int THREADS, int VECS, bool ALIGNED, bool OUT_ALIGNED, bool GT = false>
__global__ void __launch_bounds__(THREADS)
compact_kernel(const uint32_t *__restrict__ in, const uint8_t *__restrict__ flags, uint32_t *__restrict__ out,
               int32_t *__restrict__ count, size_t n, unsigned num_tiles, unsigned long long *status,
               DevState *st, unsigned capacity, unsigned spin_limit, int32_t threshold = 0)
{
    constexpr int NWARPS = THREADS / 32;
    constexpr int WARP_ITEMS = 32 * 4 * VECS;
    constexpr int TILE = THREADS * 4 * VECS;
    using B = StageBuffer<TILE>;
    __shared__ __align__(16) uint32_t s_stage_raw[B::kWords];
    __shared__ unsigned s_warp[NWARPS];
    __shared__ unsigned s_prefix;
    __shared__ unsigned s_tile;
    uint32_t *s_stage = s_stage_raw + B::kLead;
    const AddU32 op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) s_tile = atomicAdd(&st->ticket, 1u);
    __syncthreads();
    const unsigned tile = s_tile;
    if (tile >= num_tiles) return;   // never taken: each launch hands out exactly num_tiles tickets
    const size_t tile_base = static_cast<size_t>(tile) * TILE;
    const size_t warp_base = tile_base + static_cast<size_t>(warp) * WARP_ITEMS;
    const bool full = tile_base + TILE <= n;

    uint32_t x[VECS][4];
    load_rows<uint32_t, VECS, ALIGNED>(in, warp_base, n, lane, full, x, 0u);
    uint32_t keep[VECS];
    if (GT) {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            const size_t e = warp_base + static_cast<size_t>(r * 32 + lane) * 4;
            uint32_t m = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if ((full || e + k < n) && static_cast<int32_t>(x[r][k]) > threshold) m |= 1u << k;
            keep[r] = m;
        }
    } else if (ALIGNED && full) {
        uint32_t f[VECS];
#pragma unroll
        for (int r = 0; r < VECS; ++r)
            f[r] = ld_stream_u32(reinterpret_cast<const uint32_t *>(flags + warp_base) + r * 32 + lane);
#pragma unroll
        for (int r = 0; r < VECS; ++r) keep[r] = nonzero_byte_mask(f[r]);
    } else {
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            const size_t e = warp_base + static_cast<size_t>(r * 32 + lane) * 4;
            uint32_t m = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (e + k < n && flags[e + k] != 0) m |= 1u << k;
            keep[r] = m;
        }
    }

    uint32_t t[VECS];
#pragma unroll
    for (int r = 0; r < VECS; ++r) t[r] = __popc(keep[r]);
    uint32_t row_excl[VECS], warp_total;
    warp_scan_rows<AddU32, VECS>(op, t, lane, row_excl, warp_total);
    if (lane == 0) s_warp[warp] = warp_total;
    __syncthreads();
    uint32_t warp_excl, tile_total;
    block_scan_warps<AddU32, NWARPS>(op, s_warp, warp, lane, warp_excl, tile_total);

    unsigned tag = 0;
    if (warp == 0) {
        tag = __shfl_sync(kFullMask, lane == 0 ? read_tag(st) : 0u, 0);
        publish<AddU32>(status, tile, tag, tile == 0 ? kFlagInclusive : kFlagAggregate, tile_total, lane);
    }

    // stage the kept values at their tile-local rank
#pragma unroll
    for (int r = 0; r < VECS; ++r) {
        uint32_t rank = warp_excl + row_excl[r];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if ((keep[r] >> k) & 1u) {
                s_stage[rank] = x[r][k];
                ++rank;
            }
        }
    }

    if (warp == 0) {
        uint32_t prefix = 0;
        if (tile != 0) {
            prefix = lookback<AddU32, kLookbackPerLane>(op, status, tile, tag, &st->error, spin_limit, lane);
            publish<AddU32>(status, tile, tag, kFlagInclusive, prefix + tile_total, lane);
        }
        if (lane == 0) {
            s_prefix = prefix;
            if (tile == num_tiles - 1) *count = static_cast<int32_t>(prefix + tile_total);
        }
        if (tile == num_tiles - 1) finish_launch(st, status, num_tiles, capacity, lane);
    }
    __syncthreads();

    if (OUT_ALIGNED)
        write_run_aligned<THREADS, TILE>(out, s_prefix, tile_total, s_stage, 0, tid, n);
    else
        write_run_scalar<THREADS>(out, s_prefix, tile_total, s_stage, 0, tid, n);
}


// Ring depths measured on GB300 at 2^26: flags pass A (8 KB per tile) with
// 3 A and 3 B buffers; the fused predicate (32 KB per tile in both passes)
// with 2 A and 3 B buffers (100 against 114 us at 99% kept than 3 and 2).
using CompactPipe = CompactPolicy<16, 4, 4, 3, 3, 8, 1>;
using CompactGtPipe = CompactGtPolicy<16, 4, 4, 2, 3, 10, 1>;
constexpr unsigned kCompactWaitLimit = 1u << 18;
constexpr size_t kCompactPipelineMinN = size_t(1) << 19;

cudaError_t launch_compact(const int32_t *in, const uint8_t *flags, int32_t *out, int32_t *count, size_t n,
                           int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    const bool out_aligned = reinterpret_cast<uintptr_t>(out) % 16 == 0;
    const uint32_t *vin = reinterpret_cast<const uint32_t *>(in);
    uint32_t *vout = reinterpret_cast<uint32_t *>(out);
    const bool bulk_ok = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(flags) % 16 == 0);
    const bool pipelined =
        bulk_ok && (carry == kCarryPipelined || (carry != kCarryLookback && n >= kCompactPipelineMinN));
    if (pipelined) {
        using G = PipeShape<CompactPipe>;
        auto kernel = pipeline_l2_kernel<CompactPipe>;
        static std::atomic<unsigned long long> attribute_set{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const unsigned long long bit = 1ull << (dev & 63);
        if ((attribute_set.load() & bit) == 0) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(G::kSmemBytes));
            if (e != cudaSuccess) return e;
            attribute_set.fetch_or(bit);
        }
        const unsigned tiles = tiles_for(n, CompactPipe::kTile);
        const unsigned grid = tiles < static_cast<unsigned>(ws.num_sms) ? tiles : static_cast<unsigned>(ws.num_sms);
        CompactPipe::Args args{vin, flags, vout, count, n, tiles, out_aligned};
        kernel<<<grid, G::kThreads, G::kSmemBytes, s>>>(args, tiles, ws.status, ws.state, ws.capacity, spin_limit,
                                                        kCompactWaitLimit);
        return cudaGetLastError();
    }
    constexpr int THREADS = kCompactThreads, VECS = kCompactVecs;
    const unsigned tiles = tiles_for(n, kCompactTile);
    const bool aligned = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(flags) % 4 == 0);
    if (aligned && out_aligned)
        compact_kernel<THREADS, VECS, true, true><<<tiles, THREADS, 0, s>>>(
            vin, flags, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    else if (aligned)
        compact_kernel<THREADS, VECS, true, false><<<tiles, THREADS, 0, s>>>(
            vin, flags, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    else if (out_aligned)
        compact_kernel<THREADS, VECS, false, true><<<tiles, THREADS, 0, s>>>(
            vin, flags, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    else
        compact_kernel<THREADS, VECS, false, false><<<tiles, THREADS, 0, s>>>(
            vin, flags, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit);
    return cudaGetLastError();
}

template <class P>
cudaError_t set_pipeline_smem(void (*kernel)(typename P::Args, unsigned, unsigned long long *, DevState *, unsigned,
                                             unsigned, unsigned),
                              std::atomic<unsigned long long> &attribute_set)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if ((attribute_set.load() & bit) == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(PipeShape<P>::kSmemBytes));
        if (e != cudaSuccess) return e;
        attribute_set.fetch_or(bit);
    }
    return cudaSuccess;
}

cudaError_t launch_compact_gt(const int32_t *in, int32_t threshold, int32_t *out, int32_t *count, size_t n,
                              int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    const bool out_aligned = reinterpret_cast<uintptr_t>(out) % 16 == 0;
    const bool in_aligned = reinterpret_cast<uintptr_t>(in) % 16 == 0;
    const uint32_t *vin = reinterpret_cast<const uint32_t *>(in);
    uint32_t *vout = reinterpret_cast<uint32_t *>(out);
    const bool pipelined =
        in_aligned && (carry == kCarryPipelined || (carry != kCarryLookback && n >= kCompactPipelineMinN));
    if (pipelined) {
        using G = PipeShape<CompactGtPipe>;
        auto kernel = pipeline_l2_kernel<CompactGtPipe>;
        static std::atomic<unsigned long long> attribute_set{0};
        cudaError_t e = set_pipeline_smem<CompactGtPipe>(kernel, attribute_set);
        if (e != cudaSuccess) return e;
        const unsigned tiles = tiles_for(n, CompactGtPipe::kTile);
        const unsigned grid = tiles < static_cast<unsigned>(ws.num_sms) ? tiles : static_cast<unsigned>(ws.num_sms);
        CompactGtPipe::Args args{vin, threshold, vout, count, n, tiles, out_aligned};
        kernel<<<grid, G::kThreads, G::kSmemBytes, s>>>(args, tiles, ws.status, ws.state, ws.capacity, spin_limit,
                                                        kCompactWaitLimit);
        return cudaGetLastError();
    }
    constexpr int THREADS = kCompactThreads, VECS = kCompactVecs;
    const unsigned tiles = tiles_for(n, kCompactTile);
    if (in_aligned && out_aligned)
        compact_kernel<THREADS, VECS, true, true, true><<<tiles, THREADS, 0, s>>>(
            vin, nullptr, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, threshold);
    else if (in_aligned)
        compact_kernel<THREADS, VECS, true, false, true><<<tiles, THREADS, 0, s>>>(
            vin, nullptr, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, threshold);
    else if (out_aligned)
        compact_kernel<THREADS, VECS, false, true, true><<<tiles, THREADS, 0, s>>>(
            vin, nullptr, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, threshold);
    else
        compact_kernel<THREADS, VECS, false, false, true><<<tiles, THREADS, 0, s>>>(
            vin, nullptr, vout, count, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, threshold);
    return cudaGetLastError();
}

}  // namespace devscan
