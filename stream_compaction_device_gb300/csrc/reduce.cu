// Fold of a whole array into one value (sm_103a): the "reduce" step of the
// multi-block scan in geek-doc.cn "并行前缀和 scan ..." section 四 (each block
// reduces its part, the block totals are combined) and of lpnh.cn "并行扫描"
// section 3.2's multi-level scheme.  A scan split across devices needs it
// twice per shard: the shard's own total, and the fold of the totals of the
// shards before it (the shard's carry-in).
//
// One launch, one 1,024-thread block per SM.  Block b folds a contiguous
// chunk of the 16-byte-aligned body with streaming 128-bit loads, eight in
// flight per thread; the fold runs thread, warp (fixed shuffle tree), block
// (warps in order), so an fp32 sum does not depend on timing.  Each block
// hands in its total; the last block to arrive folds the block totals in
// block order, puts the (at most three) elements before the body's first
// 16-byte boundary in front, writes the result and resets the arrival
// counter.  No block waits for another.
#include "core.cuh"
#include "launch.h"

namespace devscan {
namespace {

constexpr int kReduceThreads = 1024;
constexpr int kReduceUnroll = 8;   // 16-byte loads in flight per thread

template <class Op>
__device__ __forceinline__ typename Op::S fold4(const Op &op, const uint4 &q)
{
    using S = typename Op::S;
    return op(op(from_bits<S>(q.x), from_bits<S>(q.y)), op(from_bits<S>(q.z), from_bits<S>(q.w)));
}

// Fold of v over the warp in a fixed shuffle order (every lane gets it).
template <class Op>
__device__ __forceinline__ typename Op::S warp_fold_fixed(const Op &op, typename Op::S v)
{
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
    return v;
}

// base[0 .. head) are the elements before the first 16-byte boundary; the
// body base[head .. n) is split into chunks of `chunk` elements (a multiple
// of 4), one per block.
template <class Op>
__global__ void __launch_bounds__(kReduceThreads, 1)
reduce_kernel(const typename Op::S *__restrict__ base, size_t n, unsigned head, size_t chunk,
              typename Op::S *__restrict__ block_sums, typename Op::S *__restrict__ total, DevState *st)
{
    using S = typename Op::S;
    constexpr int NW = kReduceThreads / 32;
    __shared__ S s_w[NW];
    __shared__ int s_last;
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const S *body = base + head;
    const size_t m = n - head;
    const size_t b0 = static_cast<size_t>(blockIdx.x) * chunk;
    const size_t b1 = b0 >= m ? b0 : (b0 + chunk < m ? b0 + chunk : m);   // empty past the body's end
    const uint4 *rows = reinterpret_cast<const uint4 *>(body);
    const size_t r1 = b1 / 4;   // whole 16-byte rows of the chunk end here

    S acc = Op::identity();
    size_t r = b0 / 4 + tid;
    for (; r + static_cast<size_t>(kReduceUnroll - 1) * kReduceThreads < r1; r += kReduceUnroll * kReduceThreads) {
        uint4 q[kReduceUnroll];
#pragma unroll
        for (int u = 0; u < kReduceUnroll; ++u) q[u] = ld_stream(rows + r + static_cast<size_t>(u) * kReduceThreads);
#pragma unroll
        for (int u = 0; u < kReduceUnroll; ++u) acc = op(acc, fold4(op, q[u]));
    }
    for (; r < r1; r += kReduceThreads) acc = op(acc, fold4(op, ld_stream(rows + r)));
    if (b1 > r1 * 4 && static_cast<size_t>(tid) < b1 - r1 * 4) acc = op(acc, body[r1 * 4 + tid]);   // ragged end

    acc = warp_fold_fixed(op, acc);
    if (lane == 0) s_w[warp] = acc;
    __syncthreads();
    if (tid < 32) {
        S v = s_w[lane];   // NW == 32
        v = warp_fold_fixed(op, v);
        if (lane == 0) {
            block_sums[blockIdx.x] = v;
            __threadfence();   // the total before the arrival that counts it
            s_last = atomicAdd(&st->grid_arrive, 1u) == gridDim.x - 1;
        }
    }
    __syncthreads();
    if (!s_last || warp != 0) return;
    __threadfence();
    S v = Op::identity();
    for (unsigned b = lane; b < gridDim.x; b += 32) v = op(v, __ldcg(block_sums + b));
    v = warp_fold_fixed(op, v);
    if (lane == 0) {
        if (head != 0) {
            S h = base[0];
            for (unsigned k = 1; k < head; ++k) h = op(h, base[k]);
            v = op(h, v);
        }
        *total = v;
        st->grid_arrive = 0;   // for the next launch on the stream
    }
}

template <class Op>
__global__ void write_identity_kernel(typename Op::S *total)
{
    *total = Op::identity();
}

template <class Op>
cudaError_t launch_reduce_op(const void *in, size_t n, void *total, const Workspace &ws, cudaStream_t s)
{
    using S = typename Op::S;
    S *t = static_cast<S *>(total);
    if (n == 0) {
        write_identity_kernel<Op><<<1, 1, 0, s>>>(t);
        return cudaGetLastError();
    }
    const S *base = static_cast<const S *>(in);
    const unsigned mis = static_cast<unsigned>((16 - reinterpret_cast<uintptr_t>(base) % 16) % 16) / 4;
    const unsigned head = static_cast<size_t>(mis) < n ? mis : static_cast<unsigned>(n);
    const size_t m = n - head;
    constexpr size_t kRowUnit = static_cast<size_t>(kReduceThreads) * 4;   // one row per thread
    const size_t units = (m + kRowUnit - 1) / kRowUnit;
    size_t blocks = units < static_cast<size_t>(ws.num_sms) ? units : static_cast<size_t>(ws.num_sms);
    if (blocks == 0) blocks = 1;
    const size_t chunk = units == 0 ? kRowUnit : ((units + blocks - 1) / blocks) * kRowUnit;
    blocks = m == 0 ? 1 : (m + chunk - 1) / chunk;   // every block starts inside the body
    reduce_kernel<Op><<<static_cast<unsigned>(blocks), kReduceThreads, 0, s>>>(
        base, n, head, chunk, reinterpret_cast<S *>(ws.tile_sums), t, ws.state);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reduce(ElemType type, int op, const void *in, size_t n, void *total, const Workspace &ws,
                          cudaStream_t s)
{
    switch (type) {
    case ElemType::I32:
        if (op == kOpAdd) return launch_reduce_op<AddU32>(in, n, total, ws, s);
        if (op == kOpMax) return launch_reduce_op<MaxI32>(in, n, total, ws, s);
        return launch_reduce_op<XorU32>(in, n, total, ws, s);
    case ElemType::U32:
        if (op == kOpAdd) return launch_reduce_op<AddU32>(in, n, total, ws, s);
        if (op == kOpMax) return launch_reduce_op<MaxU32>(in, n, total, ws, s);
        return launch_reduce_op<XorU32>(in, n, total, ws, s);
    case ElemType::F32:
        if (op == kOpAdd) return launch_reduce_op<AddF32>(in, n, total, ws, s);
        return launch_reduce_op<MaxF32>(in, n, total, ws, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace devscan
