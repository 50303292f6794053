// Bracket check fused into the inclusive add-scan (sm_103a).
//
// geek-doc.cn "并行前缀和 scan ..." section 一: with '(' as +1 and ')' as -1,
// one scan answers two questions -- a negative running sum means a surplus
// ')', a nonzero final sum means the brackets do not pair up.  Here both
// answers come out of the scan's own pass: every consumed tile tests its
// scanned values for a negative one (a warp vote; a warp that finds one
// stores 1 into result[0], at most once per launch) and the last tile writes
// the final sum into result[1].  The
// scanned array itself is stored only when the caller asks for it.
//
// The check alone (no scanned array wanted) needs no scan at all: a run of
// weights is summed up by (sum, lowest and highest of its own inclusive
// prefixes), and two runs combine as
//     (s1, lo1, hi1) then (s2, lo2, hi2) = (s1 + s2, min(lo1, s1 + lo2), max(hi1, s1 + hi2)),
// an associative fold.  bracket_check_kernel folds in 64-bit integers (exact
// for n < 2^31), reads the input once, meets at one grid barrier and then
// decides each chunk from its offset: the int32 prefixes are the exact ones
// modulo 2^32, and while a chunk's prefixes stay inside one window
// [k 2^32 - 2^31, k 2^32 + 2^31) the wrapped lowest prefix is the lowest
// wrapped prefix, so the chunk holds a negative one exactly when its wrapped
// lowest prefix is negative.  A chunk that spans two windows (possible only
// with large weights) is checked again element by element.
#include <atomic>

#include "core.cuh"
#include "grid_sync.cuh"
#include "launch.h"
#include "pipeline_l2.cuh"
#include "scan_kernel.cuh"

namespace devscan {
namespace {

// result[0] = 1 when any value of these scanned rows is negative (int32);
// the thread holding tid 0 of the last tile writes result[1].  Rows padded
// past n repeat the last inclusive value, so padding changes neither answer.
// `marked` (warp-uniform) remembers that this warp has stored the flag
// already: all warps storing to one word on every tile would queue up at its
// L2 slice.
template <int VECS>
__device__ __forceinline__ void bracket_mark(int32_t *result, const uint32_t (&x)[VECS][4], bool last_tile,
                                             uint32_t incl_end, int tid, int lane, unsigned &marked)
{
    int32_t lo = 0;
#pragma unroll
    for (int q = 0; q < VECS; ++q)
#pragma unroll
        for (int j = 0; j < 4; ++j) lo = min(lo, static_cast<int32_t>(x[q][j]));
    if (marked == 0 && __any_sync(kFullMask, lo < 0)) {
        if (lane == 0) result[0] = 1;
        marked = 1;
    }
    if (last_tile && tid == 0) result[1] = static_cast<int32_t>(incl_end);
}

// Epilogue of the one-tile-per-block scan kernel.
struct BracketEpilogue {
    struct Args {
        int32_t *result;
    };
    static constexpr bool kActive = true;
    template <class S, int VECS>
    __device__ static void tile(const Args &e, const S (&x)[VECS][4], bool last_tile, S incl_end, int tid, int lane)
    {
        unsigned marked = 0;   // one tile per block: nothing to remember
        bracket_mark<VECS>(e.result, x, last_tile, incl_end, tid, lane, marked);
    }
};

// Pipelined scan policy with the same epilogue (geometry of the int32 scan:
// parts folded in pass A, no barrier among the consume warps, two tiles per
// ticket).
using BracketBase = ScanPolicy<AddU32, true, 16, 4, 4, 2, 4, 10, kL2EvictLast, kL2EvictFirst, true, 1, true, 2>;

struct BracketPolicy : BracketBase {
    struct Args : BracketBase::Args {
        int32_t *result;
        unsigned num_tiles;
    };
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *, uint32_t *, int warp,
                                       int lane, Release &release)
    {
        uint32_t x[VECS][4];
        load_x(a, ct, warp, lane, x);
        const uint32_t pfx = ct.prefix + ct.part_excl[warp];
        release();   // the tile and the part's prefix are in registers now
        scan_x_from(pfx, lane, x);
        bracket_mark<VECS>(a.result, x, ct.tile == a.num_tiles - 1, ct.prefix + ct.aggregate, warp * 32 + lane, lane,
                           *ct.warp_state);
        if (a.out != nullptr) store_x(a.out, a.n, ct.tile, warp, lane, x);
        return 0;
    }
};

// ---------------------------------------------------------------------------
// Read-only check: one cooperative launch of one block per SM.
// ---------------------------------------------------------------------------
// A run of weights: its sum and the lowest / highest of its inclusive
// prefixes (an empty run has lo = +kNoPrefix, hi = -kNoPrefix).
struct Run {
    long long s, lo, hi;
};
constexpr long long kNoPrefix = 1ll << 62;   // |any prefix| < 2^62 for n < 2^31

__device__ __forceinline__ Run run_then(const Run &a, const Run &b)
{
    return Run{a.s + b.s, min(a.lo, a.s + b.lo), max(a.hi, a.s + b.hi)};
}

__device__ __forceinline__ long long shfl_up_ll(long long v, int d)
{
    return static_cast<long long>(__shfl_up_sync(kFullMask, static_cast<unsigned long long>(v), d));
}
__device__ __forceinline__ long long shfl_xor_ll(long long v, int d)
{
    return static_cast<long long>(__shfl_xor_sync(kFullMask, static_cast<unsigned long long>(v), d));
}

// The runs of the 32 lanes, in lane order, as one run (in every lane).
__device__ __forceinline__ Run warp_run(const Run &r, int lane)
{
    long long inc = r.s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const long long u = shfl_up_ll(inc, d);
        if (lane >= d) inc += u;
    }
    const long long before = inc - r.s;
    long long lo = before + r.lo, hi = before + r.hi;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        lo = min(lo, shfl_xor_ll(lo, d));
        hi = max(hi, shfl_xor_ll(hi, d));
    }
    return Run{static_cast<long long>(__shfl_sync(kFullMask, static_cast<unsigned long long>(inc), 31)), lo, hi};
}

// True when the exact prefixes p in [lo, hi] all lie in one 2^32-wide window
// centred on a multiple of 2^32 (so wrapping to int32 keeps their order).
__device__ __forceinline__ bool one_window(long long lo, long long hi)
{
    return ((lo + (1ll << 31)) >> 32) == ((hi + (1ll << 31)) >> 32);
}

constexpr int kCheckThreads = 1024;
constexpr int kCheckWarps = kCheckThreads / 32;
constexpr int kCheckSeg = 512;   // elements a warp takes per step: 16 consecutive ones per lane

// This lane's 16 consecutive weights of the segment at e0 (past `end`:
// absent, counted as 0 and not as prefixes).
__device__ __forceinline__ void load_seg16(const int32_t *__restrict__ in, size_t e0, size_t end, int lane,
                                           int32_t (&w)[16], unsigned &valid)
{
    const size_t b = e0 + static_cast<size_t>(lane) * 16;
    if (b + 16 <= end) {
        const uint4 *p = reinterpret_cast<const uint4 *>(in + b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 q = __ldcs(p + k);
            w[4 * k] = static_cast<int32_t>(q.x);
            w[4 * k + 1] = static_cast<int32_t>(q.y);
            w[4 * k + 2] = static_cast<int32_t>(q.z);
            w[4 * k + 3] = static_cast<int32_t>(q.w);
        }
        valid = 0xffffu;
    } else {
        valid = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const bool has = b + j < end;
            w[j] = has ? in[b + j] : 0;
            if (has) valid |= 1u << j;
        }
    }
}

// The run of this lane's 16 weights.
__device__ __forceinline__ Run lane_run(const int32_t (&w)[16], unsigned valid)
{
    Run r{0, kNoPrefix, -kNoPrefix};
    if (valid == 0xffffu) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            r.s += w[j];
            r.lo = min(r.lo, r.s);
            r.hi = max(r.hi, r.s);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if ((valid >> j) & 1u) {
                r.s += w[j];
                r.lo = min(r.lo, r.s);
                r.hi = max(r.hi, r.s);
            }
    }
    return r;
}

// The segment's run when every weight lies in [-2^20, 2^20) and the segment
// is whole: then every partial sum of its 512 weights fits an int32, so the
// lane folds and the warp combines in 32-bit arithmetic (one redux
// instruction each for the lowest and highest prefix).  Returns false (and
// leaves r alone) otherwise.
__device__ __forceinline__ bool warp_run_small(const int32_t (&w)[16], unsigned valid, int lane, Run &r)
{
    uint32_t span = 0;   // the largest w + 2^20, as unsigned: below 2^21 iff every w fits
#pragma unroll
    for (int j = 0; j < 16; ++j) span = max(span, static_cast<uint32_t>(w[j]) + (1u << 20));
    if (!__all_sync(kFullMask, valid == 0xffffu && span < (1u << 21))) return false;
    int32_t p = 0, lo = INT32_MAX, hi = INT32_MIN;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        p += w[j];
        lo = min(lo, p);
        hi = max(hi, p);
    }
    int32_t inc = p;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t u = __shfl_up_sync(kFullMask, inc, d);
        if (lane >= d) inc += u;
    }
    const int32_t before = inc - p;
    r.s = __shfl_sync(kFullMask, inc, 31);
    r.lo = __reduce_min_sync(kFullMask, before + lo);
    r.hi = __reduce_max_sync(kFullMask, before + hi);
    return true;
}

// Element-by-element check of the part [wb, we) whose first prefix starts
// from `carry` (wrapped int32 prefixes): true when one is negative.
__device__ bool part_has_negative(const int32_t *__restrict__ in, size_t wb, size_t we, uint32_t carry, int lane)
{
    bool neg = false;
    for (size_t e0 = wb; e0 < we; e0 += kCheckSeg) {
        int32_t w[16];
        unsigned valid;
        load_seg16(in, e0, we, lane, w, valid);
        uint32_t t = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) t += static_cast<uint32_t>(w[j]);
        uint32_t inc = t;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t u = __shfl_up_sync(kFullMask, inc, d);
            if (lane >= d) inc += u;
        }
        uint32_t p = carry + inc - t;
        bool mine = false;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            p += static_cast<uint32_t>(w[j]);
            if (((valid >> j) & 1u) && static_cast<int32_t>(p) < 0) mine = true;
        }
        neg = neg || __any_sync(kFullMask, mine);
        carry += __shfl_sync(kFullMask, inc, 31);
    }
    return neg;
}

// result[0] = 1 when a wrapped inclusive prefix is negative, result[1] = the
// last one.  Block b owns [b * chunk, (b + 1) * chunk), warp w the w-th
// 1/32 of it; runs[3 b .. 3 b + 2] hold the block's run for the others.
__global__ void __launch_bounds__(kCheckThreads, 1)
bracket_check_kernel(const int32_t *__restrict__ in, size_t n, size_t chunk, long long *__restrict__ runs,
                     int32_t *__restrict__ result, DevState *st, unsigned spin_limit)
{
    __shared__ long long s_ws[kCheckWarps], s_wlo[kCheckWarps], s_whi[kCheckWarps];
    __shared__ long long s_off;
    __shared__ int s_neg;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned blocks = gridDim.x;
    const size_t begin = static_cast<size_t>(blockIdx.x) * chunk;
    const size_t end = begin + chunk < n ? begin + chunk : n;
    const size_t wpart = chunk / kCheckWarps;
    const size_t wb = begin + static_cast<size_t>(warp) * wpart;
    const size_t we = wb + wpart < end ? wb + wpart : end;
    if (tid == 0) s_neg = 0;

    // ---- the warp's run, segment by segment (the next one loaded ahead)
    Run acc{0, kNoPrefix, -kNoPrefix};
    int32_t wn[16];
    unsigned vn = 0;
    if (wb < we) load_seg16(in, wb, we, lane, wn, vn);
    for (size_t e0 = wb; e0 < we; e0 += kCheckSeg) {
        int32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = wn[j];
        const unsigned v = vn;
        if (e0 + kCheckSeg < we) load_seg16(in, e0 + kCheckSeg, we, lane, wn, vn);
        Run r;
        if (!warp_run_small(w, v, lane, r)) r = warp_run(lane_run(w, v), lane);
        acc = run_then(acc, r);
    }
    if (lane == 0) {
        s_ws[warp] = acc.s;
        s_wlo[warp] = acc.lo;
        s_whi[warp] = acc.hi;
    }
    __syncthreads();
    if (warp == 0) {
        const Run r = warp_run(Run{s_ws[lane], s_wlo[lane], s_whi[lane]}, lane);
        if (lane == 0) {
            runs[3 * blockIdx.x] = r.s;
            runs[3 * blockIdx.x + 1] = r.lo;
            runs[3 * blockIdx.x + 2] = r.hi;
        }
    }

    const bool ok = grid_barrier(st, blocks, spin_limit);

    // ---- the block's offset; then each warp decides its part
    if (warp == 0) {
        long long off = 0;
        if (ok)
            for (unsigned b = lane; b < blockIdx.x; b += 32) off += __ldcg(runs + 3 * b);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) off += shfl_xor_ll(off, d);
        if (lane == 0) {
            s_off = off;
            if (blockIdx.x == blocks - 1) result[1] = static_cast<int32_t>(static_cast<uint32_t>(off + __ldcg(runs + 3 * blockIdx.x)));
        }
    }
    __syncthreads();
    if (ok && wb < we) {
        long long before = lane < warp ? s_ws[lane] : 0;
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) before += shfl_xor_ll(before, d);
        const long long off = s_off + before;   // exact prefix before this warp's part
        const long long lo = off + s_wlo[warp], hi = off + s_whi[warp];
        bool neg;
        if (one_window(lo, hi))
            neg = static_cast<int32_t>(static_cast<uint32_t>(lo)) < 0;
        else
            neg = part_has_negative(in, wb, we, static_cast<uint32_t>(off), lane);
        if (neg && lane == 0) s_neg = 1;
    }
    __syncthreads();
    if (tid == 0 && s_neg) result[0] = 1;
    grid_depart(st, blocks);
}

cudaError_t launch_bracket_check(const int32_t *in, int32_t *result, size_t n, const Workspace &ws,
                                 unsigned spin_limit, cudaStream_t s)
{
    constexpr size_t UNIT = static_cast<size_t>(kCheckWarps) * kCheckSeg;   // one segment per warp
    const size_t units = (n + UNIT - 1) / UNIT;
    size_t blocks = units < static_cast<size_t>(ws.num_sms) ? units : static_cast<size_t>(ws.num_sms);
    const size_t slots = static_cast<size_t>(ws.capacity) * 4 / (3 * sizeof(long long));   // runs fit tile_sums
    if (blocks > slots) blocks = slots;
    const size_t chunk = ((units + blocks - 1) / blocks) * UNIT;
    blocks = (n + chunk - 1) / chunk;
    long long *runs = reinterpret_cast<long long *>(ws.tile_sums);
    DevState *st = ws.state;
    void *args[] = {const_cast<int32_t **>(&in), &n, const_cast<size_t *>(&chunk), &runs, &result, &st, &spin_limit};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(&bracket_check_kernel),
                                       dim3(static_cast<unsigned>(blocks)), dim3(kCheckThreads), args, 0, s);
}

constexpr unsigned kBracketWaitLimit = 1u << 18;
constexpr size_t kBracketPipelineMinN = size_t(1) << 19;
// The read-only check takes the cooperative kernel from here (below, one
// launch of the one-tile kernel is as fast) up to n < 2^31 (its 64-bit folds
// are exact there).
constexpr size_t kBracketCheckMinN = size_t(1) << 17, kBracketCheckMaxN = (size_t(1) << 31) - 1;

cudaError_t launch_bracket_pipelined(const uint32_t *in, uint32_t *out, int32_t *result, size_t n,
                                     const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    using P = BracketPolicy;
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
    P::Args args;
    args.in = in;
    args.out = out;
    args.n = n;
    args.result = result;
    args.num_tiles = tiles;
    kernel<<<grid, G::kThreads, G::kSmemBytes, s>>>(args, tiles, ws.status, ws.state, ws.capacity, spin_limit,
                                                    kBracketWaitLimit);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bracket(const int32_t *in, int32_t *out, int32_t *result, size_t n, int carry,
                           const Workspace &ws, unsigned spin_limit, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(result, 0, 2 * sizeof(int32_t), s);
    if (e != cudaSuccess || n == 0) return e;
    const uint32_t *uin = reinterpret_cast<const uint32_t *>(in);
    uint32_t *uout = reinterpret_cast<uint32_t *>(out);
    const bool aligned = reinterpret_cast<uintptr_t>(in) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0;
    if (out == nullptr && aligned && n <= kBracketCheckMaxN &&
        (carry == kCarryL2Resident || (carry == kCarryDefault && n >= kBracketCheckMinN)))
        return launch_bracket_check(in, result, n, ws, spin_limit, s);
    const bool pipelined =
        aligned && (carry == kCarryPipelined || (carry != kCarryLookback && n >= kBracketPipelineMinN));
    if (pipelined) return launch_bracket_pipelined(uin, uout, result, n, ws, spin_limit, s);
    const unsigned tiles = tiles_for(n, kScanTile);
    const BracketEpilogue::Args epi{result};
    if (aligned)
        scan_lookback_kernel<AddU32, kScanThreads, kScanVecs, true, true, kUseTickets, kLookbackPerLane, 1, false,
                             BracketEpilogue><<<tiles, kScanThreads, 0, s>>>(
            uin, uout, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, epi);
    else
        scan_lookback_kernel<AddU32, kScanThreads, kScanVecs, true, false, kUseTickets, kLookbackPerLane, 1, false,
                             BracketEpilogue><<<tiles, kScanThreads, 0, s>>>(
            uin, uout, n, tiles, ws.status, ws.state, ws.capacity, spin_limit, epi);
    return cudaGetLastError();
}

}  // namespace devscan
