// Small scans in one thread-block cluster (sm_103a): inputs of up to
// kClusterMaxN elements.
//
// lpnh.cn "并行扫描" section 3.2 and geek-doc.cn "并行前缀和 scan ..." section
// 四 scan each block's tile, combine the block totals, then add each block's
// offset.  Here every block of the cluster scans its tile as the one-tile
// kernel does (thread-serial fold of its rows, 5-step shuffle scans, a scan
// of the warp totals), leaves its tile total in its own shared memory and
// meets the other blocks at a cluster barrier; warp 0 then reads the totals
// of the blocks before it straight out of their shared memory (distributed
// shared memory, `mapa` + `ld.shared::cluster`) and folds them in block
// order.  A second cluster barrier keeps every block resident until the
// later blocks have read its total.  One launch, no status words, no global
// atomics and no spin: the only waits are the hardware's cluster barriers.
#include "core.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace devscan {
namespace {

constexpr int kClusterThreads = 1024;
constexpr int kClusterVecs = 2;                                       // rows of 4 elements per lane
constexpr int kClusterTile = kClusterThreads * 4 * kClusterVecs;      // 8,192 elements per block
constexpr int kClusterBlocks = 8;                                     // the portable cluster size

__device__ __forceinline__ unsigned cluster_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every block of the cluster arrives, then waits for all:
// shared-memory writes before it are visible to the whole cluster after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The 32-bit word at the same shared-memory offset as `p` in block `rank`
// of the cluster.
__device__ __forceinline__ uint32_t ld_cluster_u32(const void *p, unsigned rank)
{
    uint32_t addr, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(p)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

template <class Op, bool INCLUSIVE, bool ALIGNED>
__global__ void __launch_bounds__(kClusterThreads, 1)
scan_cluster_kernel(const typename Op::S *__restrict__ in, typename Op::S *__restrict__ out, size_t n,
                    const typename Op::S *carry_in)
{
    using S = typename Op::S;
    constexpr int NWARPS = kClusterThreads / 32, VECS = kClusterVecs;
    constexpr int WARP_ITEMS = 32 * 4 * VECS;
    __shared__ S s_warp[NWARPS];
    __shared__ S s_total;    // this block's tile total, read by the later blocks of the cluster
    __shared__ S s_prefix;
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned rank = cluster_rank();   // the grid is one cluster: rank = block index
    const size_t tile_base = static_cast<size_t>(rank) * kClusterTile;
    const size_t warp_base = tile_base + static_cast<size_t>(warp) * WARP_ITEMS;
    const bool full = tile_base + kClusterTile <= n;

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
    if (tid == 0) s_total = tile_total;

    cluster_sync();   // every block's total is in its shared memory
    if (warp == 0) {
        // lane j < rank holds block j's total; an inclusive shuffle scan folds
        // them in block order and lane rank - 1 holds the prefix
        S v = lane < static_cast<int>(rank) ? from_bits<S>(ld_cluster_u32(&s_total, lane)) : Op::identity();
#pragma unroll
        for (int d = 1; d < kClusterBlocks; d <<= 1) {
            const S u = __shfl_up_sync(kFullMask, v, d);
            if (lane >= d) v = op(u, v);
        }
        const S prefix = __shfl_sync(kFullMask, v, rank > 0 ? rank - 1 : 0);
        if (lane == 0) {
            // a carry-in (the fold of whatever precedes the array) goes in front
            if (carry_in != nullptr)
                s_prefix = rank > 0 ? op(*carry_in, prefix) : *carry_in;
            else
                s_prefix = rank > 0 ? prefix : Op::identity();
        }
    }
    cluster_sync();   // the later blocks have read s_total; s_prefix is visible block-wide

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
    store_rows<S, VECS, ALIGNED>(out, warp_base, n, lane, full, x);
}

template <class Op, bool INCLUSIVE, bool ALIGNED>
cudaError_t launch_cluster(const void *in, void *out, size_t n, cudaStream_t s, const void *carry_in)
{
    using S = typename Op::S;
    const unsigned blocks = static_cast<unsigned>((n + kClusterTile - 1) / kClusterTile);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kClusterThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = blocks;   // one cluster spans the grid
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scan_cluster_kernel<Op, INCLUSIVE, ALIGNED>, static_cast<const S *>(in),
                              static_cast<S *>(out), n, static_cast<const S *>(carry_in));
}

template <class Op>
cudaError_t dispatch(const void *in, void *out, size_t n, bool inclusive, bool aligned, cudaStream_t s,
                     const void *c)
{
    if (inclusive)
        return aligned ? launch_cluster<Op, true, true>(in, out, n, s, c) : launch_cluster<Op, true, false>(in, out, n, s, c);
    return aligned ? launch_cluster<Op, false, true>(in, out, n, s, c) : launch_cluster<Op, false, false>(in, out, n, s, c);
}

}  // namespace

static_assert(kClusterMaxN == static_cast<size_t>(kClusterBlocks) * kClusterTile,
              "the small-scan limit is one portable cluster of tiles");

cudaError_t launch_scan_cluster(ElemType type, int op, bool inclusive, const void *in, void *out, size_t n,
                                bool aligned, cudaStream_t s, const void *carry_in)
{
    if (n == 0 || n > kClusterMaxN) return cudaErrorInvalidValue;
    switch (type) {
    case ElemType::I32:
        if (op == kOpAdd) return dispatch<AddU32>(in, out, n, inclusive, aligned, s, carry_in);
        if (op == kOpMax) return dispatch<MaxI32>(in, out, n, inclusive, aligned, s, carry_in);
        return dispatch<XorU32>(in, out, n, inclusive, aligned, s, carry_in);
    case ElemType::U32:
        if (op == kOpAdd) return dispatch<AddU32>(in, out, n, inclusive, aligned, s, carry_in);
        if (op == kOpMax) return dispatch<MaxU32>(in, out, n, inclusive, aligned, s, carry_in);
        return dispatch<XorU32>(in, out, n, inclusive, aligned, s, carry_in);
    case ElemType::F32:
        if (op == kOpAdd) return dispatch<AddF32>(in, out, n, inclusive, aligned, s, carry_in);
        return dispatch<MaxF32>(in, out, n, inclusive, aligned, s, carry_in);
    }
    return cudaErrorInvalidValue;
}

}  // namespace devscan
