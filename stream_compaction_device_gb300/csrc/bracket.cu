// Bracket check fused into the inclusive add-scan (sm_103a).
//
// geek-doc.cn "并行前缀和 scan ..." section 一: with '(' as +1 and ')' as -1,
// one scan answers two questions -- a negative running sum means a surplus
// ')', a nonzero final sum means the brackets do not pair up.  Here both
// answers come out of the scan's own pass: every consumed tile tests its
// scanned values for a negative one (a warp vote; a warp that finds one
// stores 1 into result[0], at most once per launch) and the last tile writes
// the final sum into result[1].  The
// scanned array itself is stored only when the caller asks for it, so the
// check alone reads the input once (4 bytes per element) and writes nothing
// else.
#include <atomic>

#include "core.cuh"
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

// Pipelined scan policy with the same epilogue (geometry of the int32 scan).
using BracketBase = ScanPolicy<AddU32, true, 16, 4, 4, 2, 4, 10, kL2EvictLast, kL2EvictFirst, true, 1>;

struct BracketPolicy : BracketBase {
    struct Args : BracketBase::Args {
        int32_t *result;
        unsigned num_tiles;
    };
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *wbuf0, uint32_t *wbuf1,
                                       int warp, int lane, Release &release)
    {
        uint32_t x[VECS][4];
        load_x(a, ct, warp, lane, x);
        release();   // the tile is in registers now
        const uint32_t total = scan_x(ct, wbuf0, wbuf1, warp, lane, x);
        bracket_mark<VECS>(a.result, x, ct.tile == a.num_tiles - 1, ct.prefix + total, warp * 32 + lane, lane,
                           *ct.warp_state);
        if (a.out != nullptr) store_x(a.out, a.n, ct.tile, warp, lane, x);
        return 1;
    }
};

constexpr unsigned kBracketWaitLimit = 1u << 18;
constexpr size_t kBracketPipelineMinN = size_t(1) << 19;

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
