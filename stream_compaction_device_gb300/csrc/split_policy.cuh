// One-bit split policy of the persistent two-pass pipeline (sm_103a), and the
// zero-count helper both split kernels use.
#pragma once

#include "core.cuh"
#include "pipeline_l2.cuh"
#include "stage.cuh"

namespace devscan {

__device__ __forceinline__ unsigned zeros_of(uint4 q, int bit)
{
    return 4u - (((q.x >> bit) & 1u) + ((q.y >> bit) & 1u) + ((q.z >> bit) & 1u) + ((q.w >> bit) & 1u));
}

// ---------------------------------------------------------------------------
// Pipelined split (see pipeline_l2.cuh): pass A reads the tile's keys and
// counts the keys whose bit is 0 -- the aggregate the look-back carries --
// and, inside a sort, the zeros of the next bit; pass B re-reads the keys
// (from L2), ranks them, stages the zeros and then the ones in the B buffer
// and writes two contiguous runs: zeros at the tile's prefix, ones at
// Z + (tile start - prefix).  HBM traffic: 8 bytes per key.
// ---------------------------------------------------------------------------
constexpr unsigned kBarSplitStage = 8;

template <int NS_, int NR_, int VECS_, int SA_, int SB_, int R_, int PREFETCH = 0>
struct SplitPolicy {
    using Op = AddU32;
    using S = uint32_t;
    static constexpr int kAHint = kL2EvictLast, kBHint = kL2EvictFirst, kPrefetch = PREFETCH;
    static constexpr int kConsumeWarps = NS_, kReduceWarps = NR_, kRecords = R_, kAStages = SA_, kBStages = SB_;
    static constexpr int VECS = VECS_;
    static constexpr int kWarpItems = 32 * 4 * VECS;
    static constexpr int kTile = NS_ * 32 * 4 * VECS;
    static constexpr size_t kABytes = static_cast<size_t>(kTile) * 4;
    static constexpr size_t kBBytes = static_cast<size_t>(kTile) * 4 + 64;   // keys, margin for the run copy
    static constexpr bool kHasExtra = true;
    struct Args {
        const uint32_t *keys;
        uint32_t *out;
        size_t n;
        int bit;
        const unsigned *zeros_total;
        unsigned *next_zeros;   // may be null
        int next_bit;
        bool out_aligned;
    };
    __device__ static unsigned tile_len(const Args &a, unsigned t)
    {
        const size_t rem = a.n - static_cast<size_t>(t) * kTile;
        return rem < static_cast<size_t>(kTile) ? static_cast<unsigned>(rem) : static_cast<unsigned>(kTile);
    }
    __device__ static unsigned copied(const Args &a, unsigned t) { return tile_len(a, t) & ~3u; }
    __device__ static const void *a_src(const Args &a, unsigned t) { return a.keys + static_cast<size_t>(t) * kTile; }
    __device__ static unsigned a_bytes(const Args &a, unsigned t) { return copied(a, t) * 4u; }
    __device__ static void prefetch_l2(const Args &a, unsigned t, uint64_t pol)
    {
        if (a_bytes(a, t) != 0) bulk_prefetch_l2(a_src(a, t), a_bytes(a, t), pol);
    }
    __device__ static void b_copies(const Args &a, unsigned t, const void **src, unsigned *bytes, unsigned *off)
    {
        src[0] = a.keys + static_cast<size_t>(t) * kTile;
        bytes[0] = copied(a, t) * 4u;
        off[0] = 0;
    }
    __device__ static void reduce(const Args &a, const unsigned char *abuf, unsigned t, int rtid, int nthr, S &v,
                                  unsigned &extra)
    {
        const unsigned cp = copied(a, t), len = tile_len(a, t);
        const uint4 *k4 = reinterpret_cast<const uint4 *>(abuf);
        unsigned z = 0, nz = 0;
        for (unsigned c = rtid; c < cp / 4; c += nthr) {
            const uint4 q = k4[c];
            z += zeros_of(q, a.bit);
            nz += zeros_of(q, a.next_bit);
        }
        const size_t base = static_cast<size_t>(t) * kTile;
        for (unsigned e = cp + rtid; e < len; e += nthr) {
            const uint32_t k = a.keys[base + e];
            z += ((k >> a.bit) & 1u) ? 0u : 1u;
            nz += ((k >> a.next_bit) & 1u) ? 0u : 1u;
        }
        v = z;
        extra = nz;
    }
    __device__ static void after_reduce(const Args &a, unsigned, unsigned next_zero_count)
    {
        if (a.next_zeros != nullptr && next_zero_count != 0) atomicAdd(a.next_zeros, next_zero_count);
    }
    template <class Release>
    __device__ static unsigned consume(const Args &a, const ConsumeTile<S> &ct, uint32_t *wbuf0, uint32_t *wbuf1,
                                       int warp, int lane, Release &release)
    {
        constexpr int THREADS = NS_ * 32;
        const AddU32 op;
        const unsigned t = ct.tile;
        const size_t base = static_cast<size_t>(t) * kTile;
        const int wbase = warp * kWarpItems;
        uint32_t *buf = reinterpret_cast<uint32_t *>(ct.buf);
        const unsigned len = tile_len(a, t), cp = copied(a, t);
        uint32_t x[VECS][4], zmask[VECS], cnt[VECS];
#pragma unroll
        for (int q = 0; q < VECS; ++q) {
            if (len == static_cast<unsigned>(kTile)) {
                const uint4 u = reinterpret_cast<const uint4 *>(buf + wbase)[q * 32 + lane];
                x[q][0] = u.x;
                x[q][1] = u.y;
                x[q][2] = u.z;
                x[q][3] = u.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const unsigned e = static_cast<unsigned>(wbase + (q * 32 + lane) * 4 + j);
                    x[q][j] = (e < cp) ? buf[e] : ((e < len) ? a.keys[base + e] : 0u);
                }
            }
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const unsigned e = static_cast<unsigned>(wbase + (q * 32 + lane) * 4 + j);
                if (e < len && !((x[q][j] >> a.bit) & 1u)) m |= 1u << j;
            }
            zmask[q] = m;
            cnt[q] = __popc(m);
        }
        uint32_t row_excl[VECS], warp_total;
        warp_scan_rows<AddU32, VECS>(op, cnt, lane, row_excl, warp_total);
        uint32_t warp_excl, tile_zeros;
        // the barrier inside also means every thread has read the buffer
        group_scan<AddU32, NS_>(op, warp_total, (ct.round & 1) ? wbuf1 : wbuf0, warp, lane, warp_excl, tile_zeros);
        // stage both runs in phase with their destinations (both offsets are
        // known here): zeros from word z_phase, ones from the next 16-byte
        // boundary after the zeros plus o_phase
        const size_t zeros_before = ct.prefix;
        const size_t ones_at = static_cast<size_t>(*a.zeros_total) + (base - zeros_before);
        const unsigned z_phase = a.out_aligned ? static_cast<unsigned>(zeros_before & 3) : 0u;
        const unsigned o_phase = a.out_aligned ? static_cast<unsigned>(ones_at & 3) : 0u;
        const unsigned o_base = a.out_aligned ? ((z_phase + tile_zeros + 3u) & ~3u) : tile_zeros;
#pragma unroll
        for (int q = 0; q < VECS; ++q) {
            uint32_t zr = warp_excl + row_excl[q];
            const uint32_t li0 = static_cast<uint32_t>(wbase + (q * 32 + lane) * 4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t li = li0 + j;
                if (li < len) {
                    if ((zmask[q] >> j) & 1u)
                        buf[z_phase + zr++] = x[q][j];
                    else
                        buf[o_base + o_phase + (li - zr)] = x[q][j];
                }
            }
        }
        named_sync(kBarSplitStage, THREADS);
        const int tid = warp * 32 + lane;
        if (a.out_aligned) {
            write_run_direct<THREADS>(a.out, zeros_before, tile_zeros, buf, tid, a.n);
            write_run_direct<THREADS>(a.out, ones_at, len - tile_zeros, buf + o_base, tid, a.n);
        } else {
            write_run_scalar<THREADS>(a.out, zeros_before, tile_zeros, buf, 0, tid, a.n);
            write_run_scalar<THREADS>(a.out, ones_at, len - tile_zeros, buf, static_cast<int>(tile_zeros), tid, a.n);
        }
        release();
        return 1;
    }
};

}  // namespace devscan
