// L2-resident scan for inputs that fit in L2 (sm_103a): one cooperative
// launch, one block per SM, two phases around one grid barrier.
//
// geek-doc.cn "并行前缀和 scan ..." section 四: reduce the blocks, scan the
// block totals, add the offsets -- here in a single launch.  GB300's L2
// (about 126 MB) holds the whole input of a mid-size scan (2^24 four-byte
// elements are 64 MB), so the second read of the classic reduce-then-scan is
// an L2 hit and HBM still moves 2 * n * sizeof(T) bytes.  Every warp owns a
// contiguous part of its block's chunk:
//   phase 1  each warp folds its part (loads marked evict_last, so the part
//            stays in L2); the block's total goes to block_sums[b] and the
//            warp totals stay in shared memory;
//   barrier  every block arrives at a grid-wide counter (a bounded wait that
//            records a timeout in the error word);
//   phase 2  block b folds block_sums[0 .. b) in a fixed order (its offset);
//            each warp adds the totals of the block's earlier warps, then
//            re-reads its part from L2 segment by segment (the next segment
//            loaded while this one is scanned) and scans it with a running
//            carry and streaming stores.
// There is no per-tile look-back chain and no block barrier between segments,
// so a launch costs one grid barrier and two streams over the data; the fp32
// result does not depend on timing.
#include "core.cuh"
#include "grid_sync.cuh"
#include "launch.h"

namespace devscan {
namespace {

template <class Op, bool INCLUSIVE, int THREADS, int VECS>
__global__ void __launch_bounds__(THREADS, 1)
l2_resident_scan_kernel(const typename Op::S *__restrict__ in, typename Op::S *__restrict__ out, size_t n,
                        size_t chunk, typename Op::S *__restrict__ block_sums, DevState *st, unsigned spin_limit,
                        const typename Op::S *carry_in)
{
    using S = typename Op::S;
    constexpr int NWARPS = THREADS / 32;
    constexpr int SEG = 32 * 4 * VECS;   // elements a warp moves per step (the chunk is a multiple of NWARPS * SEG)
    __shared__ S s_wtot[NWARPS];
    __shared__ S s_carry;
    const Op op;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned blocks = gridDim.x;
    const size_t begin = static_cast<size_t>(blockIdx.x) * chunk;
    const size_t end = begin + chunk < n ? begin + chunk : n;
    const size_t wpart = chunk / NWARPS;
    const size_t wb = begin + static_cast<size_t>(warp) * wpart;   // this warp's part: [wb, we)
    const size_t we = wb + wpart < end ? wb + wpart : end;

    // ---- phase 1: the part's total; its lines stay in L2
    const uint64_t keep = policy_evict_last();
    S acc = Op::identity();
    size_t s = wb;
    for (; s + 2 * SEG <= we; s += 2 * SEG) {
        uint4 q[2 * VECS];
#pragma unroll
        for (int r = 0; r < 2 * VECS; ++r) q[r] = ld_keep(reinterpret_cast<const uint4 *>(in + s) + r * 32 + lane, keep);
#pragma unroll
        for (int r = 0; r < 2 * VECS; ++r)
            acc = op(acc, op(op(from_bits<S>(q[r].x), from_bits<S>(q[r].y)), op(from_bits<S>(q[r].z), from_bits<S>(q[r].w))));
    }
    for (; s < we; s += SEG) {
        for (int r = 0; r < VECS; ++r) {
            const size_t e = s + static_cast<size_t>(r * 32 + lane) * 4;
            if (e + 4 <= we) {
                const uint4 q = ld_keep(reinterpret_cast<const uint4 *>(in + e), keep);
                acc = op(acc, op(op(from_bits<S>(q.x), from_bits<S>(q.y)), op(from_bits<S>(q.z), from_bits<S>(q.w))));
            } else {
                for (int k = 0; k < 4; ++k)
                    if (e + k < we) acc = op(acc, in[e + k]);
            }
        }
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc = op(acc, __shfl_xor_sync(kFullMask, acc, d));
    if (lane == 0) s_wtot[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        S v = lane < NWARPS ? s_wtot[lane] : Op::identity();
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
        if (lane == 0) block_sums[blockIdx.x] = v;
    }

    const bool ok = grid_barrier(st, blocks, spin_limit);

    // ---- phase 2: the block's offset, the warp's offset, then the part scanned
    if (warp == 0) {
        S v = Op::identity();
        if (ok)
            for (unsigned b = lane; b < blockIdx.x; b += 32) v = op(v, __ldcg(block_sums + b));   // through L2
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
        if (lane == 0) s_carry = carry_in != nullptr ? op(*carry_in, v) : v;
    }
    __syncthreads();
    S carry;
    {
        S v = lane < warp ? s_wtot[lane] : Op::identity();
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) v = op(v, __shfl_xor_sync(kFullMask, v, d));
        carry = op(s_carry, v);
    }
    S xn[VECS][4];
    if (wb < we) load_rows<S, VECS, true>(in, wb, we, lane, wb + SEG <= we, xn, Op::identity());
    for (s = wb; s < we; s += SEG) {
        S x[VECS][4];
#pragma unroll
        for (int r = 0; r < VECS; ++r)
#pragma unroll
            for (int k = 0; k < 4; ++k) x[r][k] = xn[r][k];
        if (s + SEG < we) load_rows<S, VECS, true>(in, s + SEG, we, lane, s + 2 * SEG <= we, xn, Op::identity());
        S tt[VECS];
#pragma unroll
        for (int r = 0; r < VECS; ++r) tt[r] = op(op(x[r][0], x[r][1]), op(x[r][2], x[r][3]));
        S row_excl[VECS], warp_total;
        warp_scan_rows<Op, VECS>(op, tt, lane, row_excl, warp_total);
#pragma unroll
        for (int r = 0; r < VECS; ++r) {
            S cur = op(carry, row_excl[r]);
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
        store_rows<S, VECS, true>(out, s, we, lane, s + SEG <= we, x);
        carry = op(carry, warp_total);
    }
    grid_depart(st, blocks);
}

template <class Op, bool INCLUSIVE, int VECS>
cudaError_t launch_l2res(const void *in, void *out, size_t n, const Workspace &ws, unsigned spin_limit,
                         cudaStream_t s, const void *carry_in)
{
    using S = typename Op::S;
    constexpr int THREADS = 1024;
    constexpr size_t UNIT = static_cast<size_t>(THREADS) * 4 * VECS;   // one segment per warp
    const size_t units = (n + UNIT - 1) / UNIT;
    size_t blocks = units < static_cast<size_t>(ws.num_sms) ? units : static_cast<size_t>(ws.num_sms);
    const size_t chunk = ((units + blocks - 1) / blocks) * UNIT;
    blocks = (n + chunk - 1) / chunk;   // no block without work
    const S *sin = static_cast<const S *>(in);
    S *sout = static_cast<S *>(out);
    S *sums = reinterpret_cast<S *>(ws.tile_sums);
    DevState *st = ws.state;
    const S *carry = static_cast<const S *>(carry_in);
    void *args[] = {&sin, &sout, &n, const_cast<size_t *>(&chunk), &sums, &st, &spin_limit, &carry};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(&l2_resident_scan_kernel<Op, INCLUSIVE, THREADS, VECS>),
                                       dim3(static_cast<unsigned>(blocks)), dim3(THREADS), args, 0, s);
}

template <class Op>
cudaError_t launch_l2res_dir(bool inclusive, const void *in, void *out, size_t n, const Workspace &ws,
                             unsigned spin_limit, cudaStream_t s, const void *carry_in)
{
    // small inputs take 4,096-element chunk units so that more blocks share them
    if (n >= (size_t(1) << 21))
        return inclusive ? launch_l2res<Op, true, 2>(in, out, n, ws, spin_limit, s, carry_in)
                         : launch_l2res<Op, false, 2>(in, out, n, ws, spin_limit, s, carry_in);
    return inclusive ? launch_l2res<Op, true, 1>(in, out, n, ws, spin_limit, s, carry_in)
                     : launch_l2res<Op, false, 1>(in, out, n, ws, spin_limit, s, carry_in);
}

}  // namespace

cudaError_t launch_scan_l2_resident(ElemType type, int op, bool inclusive, const void *in, void *out, size_t n,
                                   const Workspace &ws, unsigned spin_limit, cudaStream_t s, const void *carry_in)
{
    switch (type) {
    case ElemType::I32:
        if (op == kOpAdd) return launch_l2res_dir<AddU32>(inclusive, in, out, n, ws, spin_limit, s, carry_in);
        if (op == kOpMax) return launch_l2res_dir<MaxI32>(inclusive, in, out, n, ws, spin_limit, s, carry_in);
        return launch_l2res_dir<XorU32>(inclusive, in, out, n, ws, spin_limit, s, carry_in);
    case ElemType::U32:
        if (op == kOpAdd) return launch_l2res_dir<AddU32>(inclusive, in, out, n, ws, spin_limit, s, carry_in);
        if (op == kOpMax) return launch_l2res_dir<MaxU32>(inclusive, in, out, n, ws, spin_limit, s, carry_in);
        return launch_l2res_dir<XorU32>(inclusive, in, out, n, ws, spin_limit, s, carry_in);
    case ElemType::F32:
        if (op == kOpAdd) return launch_l2res_dir<AddF32>(inclusive, in, out, n, ws, spin_limit, s, carry_in);
        return launch_l2res_dir<MaxF32>(inclusive, in, out, n, ws, spin_limit, s, carry_in);
    }
    return cudaErrorInvalidValue;
}

}  // namespace devscan
