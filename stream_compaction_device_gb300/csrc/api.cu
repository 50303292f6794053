// C ABI of the devscan library: argument validation, the per-stream
// workspace, and dispatch to the kernels.  Declared in include/devscan.h.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/devscan.h"
#include "../../include/devscan_measure.h"
#include "core.cuh"
#include "launch.h"

namespace devscan {
namespace {

// Polls of a look-back wait before it gives up (each poll after the fourth
// sleeps 32-256 ns, so the bound is well above any legitimate wait: a
// predecessor tile only has to load and reduce its own data).
constexpr unsigned kSpinLimit = 1u << 21;

// Largest tile count a workspace may hold: its capacity doubles from 1,024
// in 64-bit arithmetic up to this power of two, so no size can wrap it.
constexpr size_t kMaxTiles = size_t(1) << 31;
constexpr size_t kMaxScanN = kMaxTiles * kScanTile;

// The inter-block carry strategy of the calling thread's calls (kCarry*),
// set only through devscan_measure_set_carry_mode (include/devscan_measure.h):
// one thread choosing a path for a measurement leaves every other thread's
// calls on the default.
thread_local int t_carry_mode = kCarryDefault;
int carry_mode() { return t_carry_mode; }

struct Slot {
    void *base = nullptr;
    size_t bytes = 0;
    Workspace ws;
    void *extra = nullptr;   // per-stream scratch of the digit sort (its histograms)
    size_t extra_bytes = 0;
};

std::mutex g_mutex;
std::map<std::pair<int, uintptr_t>, Slot> g_slots;
std::map<int, int> g_num_sms;

constexpr size_t kStateBytes = 256;

size_t layout_bytes(unsigned capacity)
{
    // state | status[capacity] | group status[capacity / 32] | never_published[2] | tile_sums[capacity]
    return kStateBytes + static_cast<size_t>(capacity) * 8 + static_cast<size_t>(capacity / 32) * 8 + 16 +
           static_cast<size_t>(capacity) * 4 + 256;
}

devscan_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DEVSCAN_OK : DEVSCAN_ERR_CUDA; }

// Finds (or grows) the workspace of (current device, stream) so that it holds
// at least `tiles` tile slots.  Growth frees the old block and allocates a
// new one stream-ordered, then zeroes it on the stream, so calls already
// queued on the stream finish with the old block first.
devscan_status acquire(cudaStream_t stream, unsigned tiles, Workspace *out)
{
    static_assert(sizeof(DevState) <= kStateBytes, "device state must fit its slot");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    auto sms = g_num_sms.find(dev);
    if (sms == g_num_sms.end()) {
        int count = 0;
        if (cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DEVSCAN_ERR_CUDA;
        sms = g_num_sms.emplace(dev, count).first;
    }
    if (tiles > kMaxTiles) return DEVSCAN_ERR_INVALID;
    Slot &slot = g_slots[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (slot.base == nullptr || slot.ws.capacity < tiles) {
        size_t cap = 1024;
        while (cap < tiles) cap *= 2;   // at most kMaxTiles = 2^31
        const unsigned capacity = static_cast<unsigned>(cap);
        const size_t bytes = layout_bytes(capacity);
        if (slot.base != nullptr) {
            if (cudaFreeAsync(slot.base, stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
            slot.base = nullptr;
        }
        void *base = nullptr;
        const cudaError_t e = cudaMallocAsync(&base, bytes, stream);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            g_slots.erase({dev, reinterpret_cast<uintptr_t>(stream)});
            return e == cudaErrorMemoryAllocation ? DEVSCAN_ERR_NOMEM : DEVSCAN_ERR_CUDA;
        }
        if (cudaMemsetAsync(base, 0, bytes, stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
        char *p = static_cast<char *>(base);
        slot.base = base;
        slot.bytes = bytes;
        slot.ws.state = reinterpret_cast<DevState *>(p);
        slot.ws.status = reinterpret_cast<unsigned long long *>(p + kStateBytes);
        slot.ws.never_published = slot.ws.status + capacity + capacity / 32;
        slot.ws.tile_sums = reinterpret_cast<uint32_t *>(slot.ws.never_published + 2);
        slot.ws.capacity = capacity;
    }
    slot.ws.num_sms = sms->second;
    *out = slot.ws;
    return DEVSCAN_OK;
}

// Per-stream scratch of at least `bytes`, grown stream-ordered like the
// workspace (the slot must exist: call acquire() first).
devscan_status acquire_extra(cudaStream_t stream, size_t bytes, void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_slots.find({dev, reinterpret_cast<uintptr_t>(stream)});
    if (it == g_slots.end()) return DEVSCAN_ERR_CUDA;
    Slot &slot = it->second;
    if (slot.extra_bytes < bytes) {
        if (slot.extra != nullptr && cudaFreeAsync(slot.extra, stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
        slot.extra = nullptr;
        slot.extra_bytes = 0;
        void *p = nullptr;
        const cudaError_t e = cudaMallocAsync(&p, bytes, stream);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e == cudaErrorMemoryAllocation ? DEVSCAN_ERR_NOMEM : DEVSCAN_ERR_CUDA;
        }
        slot.extra = p;
        slot.extra_bytes = bytes;
    }
    *out = slot.extra;
    return DEVSCAN_OK;
}

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bbytes && y < x + abytes;
}

devscan_status scan_common(ElemType type, bool inclusive, const void *in, void *out, size_t n, devscan_op op,
                           cudaStream_t stream, const void *carry_in = nullptr)
{
    if (op != DEVSCAN_OP_ADD && op != DEVSCAN_OP_MAX && op != DEVSCAN_OP_XOR) return DEVSCAN_ERR_INVALID;
    if (type == ElemType::F32 && op == DEVSCAN_OP_XOR) return DEVSCAN_ERR_UNSUPPORTED;
    if (n == 0) return DEVSCAN_OK;
    if (in == nullptr || out == nullptr) return DEVSCAN_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(in) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
        return DEVSCAN_ERR_INVALID;
    if (n > kMaxScanN) return DEVSCAN_ERR_INVALID;
    if (carry_in != nullptr &&
        (reinterpret_cast<uintptr_t>(carry_in) % 4 != 0 || overlaps(carry_in, 4, out, n * 4)))
        return DEVSCAN_ERR_INVALID;
    const unsigned tiles = tiles_for(n, kScanTile);
    Workspace ws;
    const devscan_status st = acquire(stream, tiles, &ws);
    if (st != DEVSCAN_OK) return st;
    const bool aligned = reinterpret_cast<uintptr_t>(in) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0;
    const int carry = carry_mode();
    return from_cuda(launch_scan(type, static_cast<int>(op), inclusive, in, out, n, aligned, carry, ws,
                                 kSpinLimit, stream, carry_in));
}

// Host arrays in, host array out: the input is copied into the caller's
// device buffer, scanned there into the second device buffer, and the result
// copied back, all ordered on `stream`.
devscan_status scan_host_common(ElemType type, bool inclusive, const void *h_in, void *h_out, size_t n,
                                devscan_op op, void *d_in, void *d_out, cudaStream_t stream)
{
    if (op != DEVSCAN_OP_ADD && op != DEVSCAN_OP_MAX && op != DEVSCAN_OP_XOR) return DEVSCAN_ERR_INVALID;
    if (type == ElemType::F32 && op == DEVSCAN_OP_XOR) return DEVSCAN_ERR_UNSUPPORTED;
    if (n == 0) return DEVSCAN_OK;
    if (h_in == nullptr || h_out == nullptr || d_in == nullptr || d_out == nullptr) return DEVSCAN_ERR_INVALID;
    if (n > kMaxScanN) return DEVSCAN_ERR_INVALID;
    const size_t bytes = n * 4;
    if (overlaps(d_in, bytes, d_out, bytes) && d_in != d_out) return DEVSCAN_ERR_INVALID;
    if (cudaMemcpyAsync(d_in, h_in, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    const devscan_status st = scan_common(type, inclusive, d_in, d_out, n, op, stream);
    if (st != DEVSCAN_OK) return st;
    return from_cuda(cudaMemcpyAsync(h_out, d_out, bytes, cudaMemcpyDeviceToHost, stream));
}

devscan_status reduce_common(ElemType type, const void *in, size_t n, devscan_op op, void *total,
                             cudaStream_t stream)
{
    if (op != DEVSCAN_OP_ADD && op != DEVSCAN_OP_MAX && op != DEVSCAN_OP_XOR) return DEVSCAN_ERR_INVALID;
    if (type == ElemType::F32 && op == DEVSCAN_OP_XOR) return DEVSCAN_ERR_UNSUPPORTED;
    if (total == nullptr || reinterpret_cast<uintptr_t>(total) % 4 != 0) return DEVSCAN_ERR_INVALID;
    if (n > kMaxScanN) return DEVSCAN_ERR_INVALID;
    if (n > 0 && (in == nullptr || reinterpret_cast<uintptr_t>(in) % 4 != 0 || overlaps(total, 4, in, n * 4)))
        return DEVSCAN_ERR_INVALID;
    Workspace ws;
    const devscan_status st = acquire(stream, 1, &ws);
    if (st != DEVSCAN_OK) return st;
    return from_cuda(launch_reduce(type, static_cast<int>(op), in, n, total, ws, stream));
}

devscan_status segscan_common(ElemType type, bool inclusive, const void *in, const uint8_t *heads, void *out,
                              size_t n, devscan_op op, cudaStream_t stream)
{
    if (op != DEVSCAN_OP_ADD && op != DEVSCAN_OP_MAX && op != DEVSCAN_OP_XOR) return DEVSCAN_ERR_INVALID;
    if (type == ElemType::F32 && op == DEVSCAN_OP_XOR) return DEVSCAN_ERR_UNSUPPORTED;
    if (n == 0) return DEVSCAN_OK;
    if (in == nullptr || heads == nullptr || out == nullptr) return DEVSCAN_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(in) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
        return DEVSCAN_ERR_INVALID;
    if (n > kMaxScanN) return DEVSCAN_ERR_INVALID;
    if (overlaps(heads, n, out, n * 4) || (in != out && overlaps(in, n * 4, out, n * 4))) return DEVSCAN_ERR_INVALID;
    Workspace ws;
    const devscan_status st = acquire(stream, tiles_for(n, kScanTile), &ws);
    if (st != DEVSCAN_OK) return st;
    return from_cuda(launch_segscan(type, static_cast<int>(op), inclusive, in, heads, out, n,
                                    carry_mode(), ws, kSpinLimit, stream));
}

}  // namespace
}  // namespace devscan

using namespace devscan;

extern "C" {

devscan_status scan_inclusive_i32(const int32_t *in, int32_t *out, size_t n, devscan_op op, cudaStream_t stream)
{
    return scan_common(ElemType::I32, true, in, out, n, op, stream);
}
devscan_status scan_inclusive_u32(const uint32_t *in, uint32_t *out, size_t n, devscan_op op, cudaStream_t stream)
{
    return scan_common(ElemType::U32, true, in, out, n, op, stream);
}
devscan_status scan_inclusive_f32(const float *in, float *out, size_t n, devscan_op op, cudaStream_t stream)
{
    return scan_common(ElemType::F32, true, in, out, n, op, stream);
}
devscan_status scan_exclusive_i32(const int32_t *in, int32_t *out, size_t n, devscan_op op, cudaStream_t stream)
{
    return scan_common(ElemType::I32, false, in, out, n, op, stream);
}
devscan_status scan_exclusive_u32(const uint32_t *in, uint32_t *out, size_t n, devscan_op op, cudaStream_t stream)
{
    return scan_common(ElemType::U32, false, in, out, n, op, stream);
}
devscan_status scan_exclusive_f32(const float *in, float *out, size_t n, devscan_op op, cudaStream_t stream)
{
    return scan_common(ElemType::F32, false, in, out, n, op, stream);
}

devscan_status scan_inclusive_carry_i32(const int32_t *in, int32_t *out, size_t n, devscan_op op,
                                        const int32_t *carry_in, cudaStream_t stream)
{
    return scan_common(ElemType::I32, true, in, out, n, op, stream, carry_in);
}
devscan_status scan_inclusive_carry_u32(const uint32_t *in, uint32_t *out, size_t n, devscan_op op,
                                        const uint32_t *carry_in, cudaStream_t stream)
{
    return scan_common(ElemType::U32, true, in, out, n, op, stream, carry_in);
}
devscan_status scan_inclusive_carry_f32(const float *in, float *out, size_t n, devscan_op op, const float *carry_in,
                                        cudaStream_t stream)
{
    return scan_common(ElemType::F32, true, in, out, n, op, stream, carry_in);
}
devscan_status scan_exclusive_carry_i32(const int32_t *in, int32_t *out, size_t n, devscan_op op,
                                        const int32_t *carry_in, cudaStream_t stream)
{
    return scan_common(ElemType::I32, false, in, out, n, op, stream, carry_in);
}
devscan_status scan_exclusive_carry_u32(const uint32_t *in, uint32_t *out, size_t n, devscan_op op,
                                        const uint32_t *carry_in, cudaStream_t stream)
{
    return scan_common(ElemType::U32, false, in, out, n, op, stream, carry_in);
}
devscan_status scan_exclusive_carry_f32(const float *in, float *out, size_t n, devscan_op op, const float *carry_in,
                                        cudaStream_t stream)
{
    return scan_common(ElemType::F32, false, in, out, n, op, stream, carry_in);
}

devscan_status scan_inclusive_host_i32(const int32_t *h_in, int32_t *h_out, size_t n, devscan_op op, int32_t *d_in,
                                       int32_t *d_out, cudaStream_t stream)
{
    return scan_host_common(ElemType::I32, true, h_in, h_out, n, op, d_in, d_out, stream);
}
devscan_status scan_inclusive_host_u32(const uint32_t *h_in, uint32_t *h_out, size_t n, devscan_op op,
                                       uint32_t *d_in, uint32_t *d_out, cudaStream_t stream)
{
    return scan_host_common(ElemType::U32, true, h_in, h_out, n, op, d_in, d_out, stream);
}
devscan_status scan_inclusive_host_f32(const float *h_in, float *h_out, size_t n, devscan_op op, float *d_in,
                                       float *d_out, cudaStream_t stream)
{
    return scan_host_common(ElemType::F32, true, h_in, h_out, n, op, d_in, d_out, stream);
}
devscan_status scan_exclusive_host_i32(const int32_t *h_in, int32_t *h_out, size_t n, devscan_op op, int32_t *d_in,
                                       int32_t *d_out, cudaStream_t stream)
{
    return scan_host_common(ElemType::I32, false, h_in, h_out, n, op, d_in, d_out, stream);
}
devscan_status scan_exclusive_host_u32(const uint32_t *h_in, uint32_t *h_out, size_t n, devscan_op op,
                                       uint32_t *d_in, uint32_t *d_out, cudaStream_t stream)
{
    return scan_host_common(ElemType::U32, false, h_in, h_out, n, op, d_in, d_out, stream);
}
devscan_status scan_exclusive_host_f32(const float *h_in, float *h_out, size_t n, devscan_op op, float *d_in,
                                       float *d_out, cudaStream_t stream)
{
    return scan_host_common(ElemType::F32, false, h_in, h_out, n, op, d_in, d_out, stream);
}

devscan_status reduce_i32(const int32_t *in, size_t n, devscan_op op, int32_t *total, cudaStream_t stream)
{
    return reduce_common(ElemType::I32, in, n, op, total, stream);
}
devscan_status reduce_u32(const uint32_t *in, size_t n, devscan_op op, uint32_t *total, cudaStream_t stream)
{
    return reduce_common(ElemType::U32, in, n, op, total, stream);
}
devscan_status reduce_f32(const float *in, size_t n, devscan_op op, float *total, cudaStream_t stream)
{
    return reduce_common(ElemType::F32, in, n, op, total, stream);
}

devscan_status segmented_scan_inclusive_i32(const int32_t *in, const uint8_t *heads, int32_t *out, size_t n,
                                            devscan_op op, cudaStream_t stream)
{
    return segscan_common(ElemType::I32, true, in, heads, out, n, op, stream);
}
devscan_status segmented_scan_inclusive_u32(const uint32_t *in, const uint8_t *heads, uint32_t *out, size_t n,
                                            devscan_op op, cudaStream_t stream)
{
    return segscan_common(ElemType::U32, true, in, heads, out, n, op, stream);
}
devscan_status segmented_scan_inclusive_f32(const float *in, const uint8_t *heads, float *out, size_t n,
                                            devscan_op op, cudaStream_t stream)
{
    return segscan_common(ElemType::F32, true, in, heads, out, n, op, stream);
}
devscan_status segmented_scan_exclusive_i32(const int32_t *in, const uint8_t *heads, int32_t *out, size_t n,
                                            devscan_op op, cudaStream_t stream)
{
    return segscan_common(ElemType::I32, false, in, heads, out, n, op, stream);
}
devscan_status segmented_scan_exclusive_u32(const uint32_t *in, const uint8_t *heads, uint32_t *out, size_t n,
                                            devscan_op op, cudaStream_t stream)
{
    return segscan_common(ElemType::U32, false, in, heads, out, n, op, stream);
}
devscan_status segmented_scan_exclusive_f32(const float *in, const uint8_t *heads, float *out, size_t n,
                                            devscan_op op, cudaStream_t stream)
{
    return segscan_common(ElemType::F32, false, in, heads, out, n, op, stream);
}

devscan_status compact_i32(const int32_t *in, const uint8_t *flags, int32_t *out, int32_t *count, size_t n,
                           cudaStream_t stream)
{
    if (count == nullptr) return DEVSCAN_ERR_INVALID;
    if (n > static_cast<size_t>(INT32_MAX)) return DEVSCAN_ERR_INVALID;
    if (n > 0) {
        if (in == nullptr || flags == nullptr || out == nullptr) return DEVSCAN_ERR_INVALID;
        if (reinterpret_cast<uintptr_t>(in) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0 ||
            reinterpret_cast<uintptr_t>(count) % 4 != 0)
            return DEVSCAN_ERR_INVALID;
        if (overlaps(out, n * 4, in, n * 4) || overlaps(out, n * 4, flags, n) || overlaps(count, 4, out, n * 4) ||
            overlaps(count, 4, in, n * 4) || overlaps(count, 4, flags, n))
            return DEVSCAN_ERR_INVALID;
    }
    if (n == 0) return from_cuda(cudaMemsetAsync(count, 0, sizeof(int32_t), stream));
    const unsigned tiles = tiles_for(n, kCompactTile);
    Workspace ws;
    devscan_status st = acquire(stream, tiles, &ws);
    if (st != DEVSCAN_OK) return st;
    const int carry = carry_mode();
    void *part_words = nullptr;   // the two-launch path's part counts and offsets
    if (carry == kCarryL2Resident || (carry == kCarryDefault && n >= kCompactTwoPassMinN)) {
        st = acquire_extra(stream, compact_part_words(n) * sizeof(uint32_t), &part_words);
        if (st != DEVSCAN_OK) return st;
    }
    return from_cuda(launch_compact(in, flags, out, count, n, carry, ws, kSpinLimit, stream,
                                    static_cast<uint32_t *>(part_words)));
}

devscan_status compact_gt_i32(const int32_t *in, int32_t threshold, int32_t *out, int32_t *count, size_t n,
                              cudaStream_t stream)
{
    if (count == nullptr || reinterpret_cast<uintptr_t>(count) % 4 != 0) return DEVSCAN_ERR_INVALID;
    if (n > static_cast<size_t>(INT32_MAX)) return DEVSCAN_ERR_INVALID;
    if (n > 0) {
        if (in == nullptr || out == nullptr) return DEVSCAN_ERR_INVALID;
        if (reinterpret_cast<uintptr_t>(in) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
            return DEVSCAN_ERR_INVALID;
        if (overlaps(out, n * 4, in, n * 4) || overlaps(count, 4, out, n * 4) || overlaps(count, 4, in, n * 4))
            return DEVSCAN_ERR_INVALID;
    }
    if (n == 0) return from_cuda(cudaMemsetAsync(count, 0, sizeof(int32_t), stream));
    Workspace ws;
    devscan_status st = acquire(stream, tiles_for(n, kCompactTile), &ws);
    if (st != DEVSCAN_OK) return st;
    const int carry = carry_mode();
    void *part_words = nullptr;   // the two-launch path's part masks, counts and offsets
    if (carry == kCarryL2Resident) {
        st = acquire_extra(stream, compact_part_words(n) * sizeof(uint32_t), &part_words);
        if (st != DEVSCAN_OK) return st;
    }
    return from_cuda(launch_compact_gt(in, threshold, out, count, n, carry, ws, kSpinLimit, stream,
                                       static_cast<uint32_t *>(part_words)));
}

devscan_status bracket_scan_i32(const int32_t *in, int32_t *out, int32_t *result, size_t n, cudaStream_t stream)
{
    if (result == nullptr || reinterpret_cast<uintptr_t>(result) % 4 != 0) return DEVSCAN_ERR_INVALID;
    if (n > kMaxScanN) return DEVSCAN_ERR_INVALID;
    if (n > 0) {
        if (in == nullptr || reinterpret_cast<uintptr_t>(in) % 4 != 0) return DEVSCAN_ERR_INVALID;
        if (out != nullptr && reinterpret_cast<uintptr_t>(out) % 4 != 0) return DEVSCAN_ERR_INVALID;
        if (overlaps(result, 8, in, n * 4) || (out != nullptr && overlaps(result, 8, out, n * 4)))
            return DEVSCAN_ERR_INVALID;
    }
    Workspace ws;
    if (n > 0) {
        const devscan_status st = acquire(stream, tiles_for(n, kScanTile), &ws);
        if (st != DEVSCAN_OK) return st;
    }
    return from_cuda(launch_bracket(in, out, result, n, carry_mode(), ws,
                                    kSpinLimit, stream));
}

devscan_status split_bit_u32(const uint32_t *keys, uint32_t *out, int bit, size_t n, cudaStream_t stream)
{
    if (bit < 0 || bit > 31) return DEVSCAN_ERR_INVALID;
    if (n > static_cast<size_t>(INT32_MAX)) return DEVSCAN_ERR_INVALID;
    if (n == 0) return DEVSCAN_OK;
    if (keys == nullptr || out == nullptr) return DEVSCAN_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(keys) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
        return DEVSCAN_ERR_INVALID;
    if (overlaps(keys, n * 4, out, n * 4)) return DEVSCAN_ERR_INVALID;
    const unsigned tiles = tiles_for(n, kSplitTile);
    Workspace ws;
    devscan_status st = acquire(stream, tiles, &ws);
    if (st != DEVSCAN_OK) return st;
    unsigned *z = &ws.state->zeros[40];
    const int carry = carry_mode();
    if (reinterpret_cast<uintptr_t>(keys) % 16 == 0 &&
        (carry == kCarryL2Resident || (carry == kCarryDefault && n >= kSplitTwoPassMinN))) {
        void *part_words = nullptr;   // the parts' zero offsets
        st = acquire_extra(stream, split_part_words(n) * sizeof(uint32_t), &part_words);
        if (st != DEVSCAN_OK) return st;
        return from_cuda(launch_split_two_pass(keys, out, n, bit, z, static_cast<uint32_t *>(part_words), ws, stream));
    }
    if (cudaMemsetAsync(z, 0, sizeof(unsigned), stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    cudaError_t e = launch_count_zeros(keys, n, bit, z, ws, stream);
    if (e != cudaSuccess) return DEVSCAN_ERR_CUDA;
    return from_cuda(launch_split(keys, out, n, bit, z, nullptr, carry, ws, kSpinLimit, stream));
}

devscan_status radix_sort_u32(uint32_t *keys, uint32_t *tmp, size_t n, cudaStream_t stream)
{
    if (n > static_cast<size_t>(INT32_MAX)) return DEVSCAN_ERR_INVALID;
    if (n == 0) return DEVSCAN_OK;
    if (keys == nullptr || tmp == nullptr) return DEVSCAN_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(keys) % 4 != 0 || reinterpret_cast<uintptr_t>(tmp) % 4 != 0)
        return DEVSCAN_ERR_INVALID;
    if (overlaps(keys, n * 4, tmp, n * 4)) return DEVSCAN_ERR_INVALID;
    const unsigned tiles = tiles_for(n, kSplitTile);
    Workspace ws;
    devscan_status st = acquire(stream, tiles, &ws);
    if (st != DEVSCAN_OK) return st;
    unsigned *z = ws.state->zeros;   // z[b] = zero count of bit b
    const int carry = carry_mode();
    if (reinterpret_cast<uintptr_t>(keys) % 16 == 0 && reinterpret_cast<uintptr_t>(tmp) % 16 == 0 &&
        (carry == kCarryL2Resident || (carry == kCarryDefault && n >= kSortTwoPassMinN))) {
        void *part_words = nullptr;   // the parts' offsets, then the next pass's part counts
        st = acquire_extra(stream, sort_part_words(n) * sizeof(uint32_t), &part_words);
        if (st != DEVSCAN_OK) return st;
        return from_cuda(launch_sort_two_pass(keys, tmp, n, &z[40], static_cast<uint32_t *>(part_words), ws, stream));
    }
    if (cudaMemsetAsync(z, 0, 33 * sizeof(unsigned), stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    if (launch_count_zeros(keys, n, 0, &z[0], ws, stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    uint32_t *src = keys, *dst = tmp;
    for (int bit = 0; bit < 32; ++bit) {
        unsigned *next = (bit < 31) ? &z[bit + 1] : nullptr;
        if (launch_split(src, dst, n, bit, &z[bit], next, carry, ws, kSpinLimit, stream) != cudaSuccess)
            return DEVSCAN_ERR_CUDA;
        std::swap(src, dst);
    }
    return DEVSCAN_OK;
}

devscan_status radix_sort_digits_u32(uint32_t *keys, uint32_t *tmp, size_t n, cudaStream_t stream)
{
    if (n > static_cast<size_t>(INT32_MAX)) return DEVSCAN_ERR_INVALID;
    if (n == 0) return DEVSCAN_OK;
    if (keys == nullptr || tmp == nullptr) return DEVSCAN_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(keys) % 4 != 0 || reinterpret_cast<uintptr_t>(tmp) % 4 != 0)
        return DEVSCAN_ERR_INVALID;
    if (overlaps(keys, n * 4, tmp, n * 4)) return DEVSCAN_ERR_INVALID;
    const size_t hist_words = radix_hist_words(n);
    Workspace ws;
    devscan_status st = acquire(stream, tiles_for(hist_words, kScanTile), &ws);
    if (st != DEVSCAN_OK) return st;
    void *hist = nullptr;
    st = acquire_extra(stream, hist_words * sizeof(uint32_t), &hist);
    if (st != DEVSCAN_OK) return st;
    uint32_t *src = keys, *dst = tmp;
    for (int pass = 0; pass < kRadixPasses; ++pass) {
        if (launch_radix_pass(src, dst, n, pass, static_cast<uint32_t *>(hist), ws, kSpinLimit, stream) != cudaSuccess)
            return DEVSCAN_ERR_CUDA;
        std::swap(src, dst);
    }
    return DEVSCAN_OK;
}

devscan_status devscan_device_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    DevState *state = nullptr;
    void *base = nullptr;
    size_t bytes = 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = g_slots.find({dev, reinterpret_cast<uintptr_t>(stream)});
        if (it == g_slots.end()) return DEVSCAN_OK;
        state = it->second.ws.state;
        base = it->second.base;
        bytes = it->second.bytes;
    }
    unsigned err = 0;
    if (cudaMemcpy(&err, &state->error, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DEVSCAN_ERR_CUDA;
    // A launch that gave up may have left its tile counter, epoch and status
    // words half-way; the stream is idle now, so start the workspace afresh.
    if (err != 0 && cudaMemset(base, 0, bytes) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    return (err & kErrTimeout) ? DEVSCAN_ERR_TIMEOUT : DEVSCAN_OK;
}

const char *devscan_status_string(devscan_status status)
{
    switch (status) {
    case DEVSCAN_OK: return "ok";
    case DEVSCAN_ERR_INVALID: return "invalid argument";
    case DEVSCAN_ERR_UNSUPPORTED: return "operator not supported for this element type";
    case DEVSCAN_ERR_CUDA: return "CUDA runtime error";
    case DEVSCAN_ERR_TIMEOUT: return "inter-block wait timed out on the device";
    case DEVSCAN_ERR_NOMEM: return "out of device memory for the workspace";
    }
    return "unknown status";
}

devscan_status devscan_stream_release(cudaStream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_slots.find({dev, reinterpret_cast<uintptr_t>(stream)});
    if (it == g_slots.end()) return DEVSCAN_OK;
    void *base = it->second.base;
    void *extra = it->second.extra;
    g_slots.erase(it);
    if (extra != nullptr && cudaFreeAsync(extra, stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    return from_cuda(cudaFreeAsync(base, stream));
}

devscan_status devscan_measure_set_carry_mode(int mode)
{
    if (mode != kCarryDefault && mode != kCarryLookback && mode != kCarryReduceThenScan && mode != kCarryPipelined &&
        mode != kCarryL2Resident)
        return DEVSCAN_ERR_INVALID;
    t_carry_mode = mode;
    return DEVSCAN_OK;
}

devscan_status devscan_selftest_stalled_wait(unsigned int spin_limit, cudaStream_t stream)
{
    if (spin_limit == 0) return DEVSCAN_ERR_INVALID;
    Workspace ws;
    const devscan_status st = acquire(stream, 1, &ws);
    if (st != DEVSCAN_OK) return st;
    return from_cuda(launch_stalled_wait(ws, spin_limit, stream));
}

}  // extern "C"
