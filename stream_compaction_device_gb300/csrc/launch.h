// Internal host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; the public interface is include/devscan.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace devscan {

struct DevState;

// Tile geometry of the scan, compaction and split kernels: THREADS threads,
// each holding VECS rows of four 32-bit elements.
constexpr int kScanThreads = 256;
constexpr int kScanVecs = 4;
constexpr int kScanTile = kScanThreads * 4 * kScanVecs;   // 4096 elements
constexpr int kCompactThreads = 256;
constexpr int kCompactVecs = 4;
constexpr int kCompactTile = kCompactThreads * 4 * kCompactVecs;
constexpr int kSplitThreads = 256;
constexpr int kSplitVecs = 4;
constexpr int kSplitTile = kSplitThreads * 4 * kSplitVecs;
constexpr int kMaxTile = 4096;   // largest of the three (workspace sizing)

// Tile order: true = an atomic ticket hands out tile indices in the order
// blocks start (forward progress does not depend on the order in which the
// hardware dispatches blocks); false = blockIdx.x.
constexpr bool kUseTickets = true;

constexpr int kOpAdd = 0, kOpMax = 1, kOpXor = 2;
constexpr int kCarryDefault = 0, kCarryLookback = 1, kCarryReduceThenScan = 2, kCarryPipelined = 3,
              kCarryL2Resident = 4;

enum class ElemType { I32, U32, F32 };

// Per-(device, stream) scratch, carved from one allocation:
//   state           DevState (epoch, ticket, error word, zero counts)
//   status          `capacity` 8-byte tile status words, followed by
//                   capacity / 32 group status words (capacity is a power of
//                   two, at least 1024)
//   never_published 2 words kept at zero (bounded-wait self-test)
//   tile_sums       `capacity` 4-byte tile totals (reduce-then-scan)
struct Workspace {
    DevState *state = nullptr;
    unsigned long long *status = nullptr;
    unsigned long long *never_published = nullptr;
    uint32_t *tile_sums = nullptr;
    unsigned capacity = 0;
    int num_sms = 0;
};

inline unsigned tiles_for(size_t n, int tile)
{
    return static_cast<unsigned>((n + static_cast<size_t>(tile) - 1) / static_cast<size_t>(tile));
}

// carry_in: a device element folded in front of the array (tile 0's prefix),
// or null for the operator's identity.
cudaError_t launch_scan(ElemType type, int op, bool inclusive, const void *in, void *out, size_t n,
                        bool aligned, int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s,
                        const void *carry_in = nullptr);

cudaError_t launch_stalled_wait(const Workspace &ws, unsigned spin_limit, cudaStream_t s);

// `carry` (kCarry*): the pipelined kernel for kCarryPipelined, the one-tile
// kernel for kCarryLookback, the measured size threshold otherwise.
// part_words: compact_part_words(n) words of per-stream scratch for the
// two-launch path (taken, for 16-byte-aligned values and flags, from
// kCompactTwoPassMinN elements and in carry mode 4), or null.  Measured on
// GB300: it beats the pipeline from 2^23 (at 2^26: 54 against 74 us at 1%
// kept, 82 against 85 at 50%, 103 against 106 at 99%) and loses below to its
// second launch.
constexpr size_t kCompactTwoPassMinN = size_t(1) << 23;
size_t compact_part_words(size_t n);
cudaError_t launch_compact(const int32_t *in, const uint8_t *flags, int32_t *out, int32_t *count, size_t n,
                           int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s,
                           uint32_t *part_words = nullptr);

// Zero count of bit `bit` over keys[0, n) added into *zeros (which the caller
// has cleared).
cudaError_t launch_count_zeros(const uint32_t *keys, size_t n, int bit, unsigned *zeros, const Workspace &ws,
                               cudaStream_t s);

// A standalone split in two launches: zeros counted per 1,024-key part (their
// offsets and the total into *zeros), then a warp per part writes its runs;
// part_words: split_part_words(n) words of per-stream scratch.  Taken for
// 16-byte-aligned keys from kSplitTwoPassMinN keys and in carry mode 4;
// measured on GB300 it beats the count pass plus the pipelined split at every
// size from 2^20 (131 against 170 us at 2^26).
constexpr size_t kSplitTwoPassMinN = size_t(1) << 20;
size_t split_part_words(size_t n);
cudaError_t launch_split_two_pass(const uint32_t *keys, uint32_t *out, size_t n, int bit, unsigned *zeros,
                                  uint32_t *part_words, const Workspace &ws, cudaStream_t s);

// The 32-pass LSD sort from the two-launch split: one zero count of bit 0,
// then per bit a write launch that also counts the next bit's zeros per
// 1,024-key part of its output (at most four global atomics per part) and a
// small launch turning those counts into the next pass's offsets.  Measured
// on GB300 at 2^26 keys: 2.85 ms against 4.15 ms for the pipelined splits.  keys and
// tmp 16-byte aligned; the sorted keys end in `keys`; part_words:
// sort_part_words(n) words of per-stream scratch; *zeros: a device word.
// Taken from kSortTwoPassMinN keys (default or carry mode 4).
constexpr size_t kSortTwoPassMinN = size_t(1) << 20;
size_t sort_part_words(size_t n);
cudaError_t launch_sort_two_pass(uint32_t *keys, uint32_t *tmp, size_t n, unsigned *zeros, uint32_t *part_words,
                                 const Workspace &ws, cudaStream_t s);

// One split pass by bit `bit` given the total zero count *zeros.  When
// next_zeros is not null, the pass also adds the zero count of bit
// `bit + 1` into *next_zeros.
cudaError_t launch_split(const uint32_t *keys, uint32_t *out, size_t n, int bit, const unsigned *zeros,
                         unsigned *next_zeros, int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s);

// Compaction keeping in[i] when in[i] > threshold (signed), predicate
// evaluated in the kernel.
// part_words (compact_part_words(n) words, or null): the two-launch form,
// taken in carry mode 4 for 16-byte-aligned values.
cudaError_t launch_compact_gt(const int32_t *in, int32_t threshold, int32_t *out, int32_t *count, size_t n,
                              int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s,
                              uint32_t *part_words = nullptr);
// Inclusive int32 add-scan (stored when out != nullptr) with the bracket
// answers in result[0..1]; clears result first (stream-ordered).
cudaError_t launch_bracket(const int32_t *in, int32_t *out, int32_t *result, size_t n, int carry,
                           const Workspace &ws, unsigned spin_limit, cudaStream_t s);

// Scan of at most kClusterMaxN elements by one thread-block cluster (8
// blocks of 8,192 elements at most), combining the block totals through
// distributed shared memory; any 4-byte alignment.  The default below
// kClusterMaxN + 1 elements.
constexpr size_t kClusterMaxN = size_t(1) << 16;
cudaError_t launch_scan_cluster(ElemType type, int op, bool inclusive, const void *in, void *out, size_t n,
                                bool aligned, cudaStream_t s, const void *carry_in = nullptr);

// Scan of an input that fits in L2: one cooperative launch, one block per SM
// (16-byte-aligned in/out).
cudaError_t launch_scan_l2_resident(ElemType type, int op, bool inclusive, const void *in, void *out, size_t n,
                                   const Workspace &ws, unsigned spin_limit, cudaStream_t s,
                                   const void *carry_in = nullptr);

// Segmented scan: heads[i] != 0 starts a segment at i.
cudaError_t launch_segscan(ElemType type, int op, bool inclusive, const void *in, const uint8_t *heads, void *out,
                           size_t n, int carry, const Workspace &ws, unsigned spin_limit, cudaStream_t s);

// Fold of in[0, n) under `op` into the device element *total (the identity
// when n == 0); one launch, deterministic order.
cudaError_t launch_reduce(ElemType type, int op, const void *in, size_t n, void *total, const Workspace &ws,
                          cudaStream_t s);

// Digit width and passes of the multi-bit LSD radix sort.
constexpr int kRadixDigitBits = 8, kRadixPasses = 32 / kRadixDigitBits;

// One LSD radix pass (digit `pass`, bits kRadixDigitBits * pass and up) from
// src to dst; `hist` holds radix_hist_words(n) words of scratch.
cudaError_t launch_radix_pass(const uint32_t *src, uint32_t *dst, size_t n, int pass, uint32_t *hist,
                              const Workspace &ws, unsigned spin_limit, cudaStream_t s);
size_t radix_hist_words(size_t n);

}  // namespace devscan
