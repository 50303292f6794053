// Allocation-free int32 exclusive scan (see scan_exclusive_i32_noalloc in
// include/devscan.h for who needs it).
//
// The single-pass look-back scan needs scratch memory beyond its input and
// output: a device state block (epoch, tile ticket, error word) and one
// 8-byte status word per tile.  The regular entry points allocate that
// per stream; this variant keeps it in one fixed array compiled into the
// library, so it never allocates.  In host code the array's name is only a
// host-side stand-in, so its device address is looked up once per device
// with cudaGetSymbolAddress and passed to the kernel.
#include <mutex>

#include "../../include/devscan.h"
#include "core.cuh"
#include "launch.h"
#include "scan_kernel.cuh"

namespace devscan {

// Room for DEVSCAN_NOALLOC_MAX_N elements: 65,536 tiles of 4,096.
constexpr unsigned kNoAllocTiles = static_cast<unsigned>(DEVSCAN_NOALLOC_MAX_N / kScanTile);
constexpr size_t kNoAllocStateBytes = 256;
// tile status words, then one group status word per 32 tiles
constexpr size_t kNoAllocBytes =
    kNoAllocStateBytes + static_cast<size_t>(kNoAllocTiles) * 8 + static_cast<size_t>(kNoAllocTiles / 32) * 8;
static_assert(DEVSCAN_NOALLOC_MAX_N % kScanTile == 0, "whole tiles");
static_assert(kNoAllocTiles % 32 == 0, "whole groups of tiles");
static_assert(sizeof(DevState) <= kNoAllocStateBytes, "state block fits");

// The scratch: zero at module load (zero status words read as "not ready";
// epoch 0 is tag 1).  528 KiB + 256 B per device, held until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once.
cudaError_t noalloc_scratch(int dev, void **ptr)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return cudaSuccess;
}

template <class Op>
cudaError_t launch_noalloc(const int32_t *in, int32_t *out, size_t n, const Workspace &ws, cudaStream_t s)
{
    using S = typename Op::S;
    const unsigned tiles = tiles_for(n, kScanTile);
    const bool aligned = reinterpret_cast<uintptr_t>(in) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0;
    const S *vin = reinterpret_cast<const S *>(in);
    S *vout = reinterpret_cast<S *>(out);
    constexpr unsigned kSpin = 1u << 21;
    if (aligned)
        scan_lookback_kernel<Op, kScanThreads, kScanVecs, false, true, kUseTickets><<<tiles, kScanThreads, 0, s>>>(
            vin, vout, n, tiles, ws.status, ws.state, ws.capacity, kSpin);
    else
        scan_lookback_kernel<Op, kScanThreads, kScanVecs, false, false, kUseTickets><<<tiles, kScanThreads, 0, s>>>(
            vin, vout, n, tiles, ws.status, ws.state, ws.capacity, kSpin);
    return cudaGetLastError();
}

}  // namespace
}  // namespace devscan

using namespace devscan;

extern "C" devscan_status scan_exclusive_i32_noalloc(const int32_t *in, int32_t *out, size_t n, devscan_op op,
                                                     cudaStream_t stream)
{
    if (op != DEVSCAN_OP_ADD && op != DEVSCAN_OP_MAX && op != DEVSCAN_OP_XOR) return DEVSCAN_ERR_INVALID;
    if (n == 0) return DEVSCAN_OK;
    if (n > DEVSCAN_NOALLOC_MAX_N) return DEVSCAN_ERR_INVALID;
    if (in == nullptr || out == nullptr) return DEVSCAN_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(in) % 4 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0)
        return DEVSCAN_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DEVSCAN_ERR_CUDA;
    void *base = nullptr;
    if (noalloc_scratch(dev, &base) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    Workspace ws;
    ws.state = static_cast<DevState *>(base);
    ws.status = reinterpret_cast<unsigned long long *>(static_cast<char *>(base) + kNoAllocStateBytes);
    ws.capacity = kNoAllocTiles;
    // the tile counter must start at zero (each launch's last tile also
    // resets it; clearing here covers a launch that never ran)
    if (cudaMemsetAsync(&ws.state->ticket, 0, sizeof(unsigned), stream) != cudaSuccess) return DEVSCAN_ERR_CUDA;
    cudaError_t e;
    if (op == DEVSCAN_OP_ADD)
        e = launch_noalloc<AddU32>(in, out, n, ws, stream);
    else if (op == DEVSCAN_OP_MAX)
        e = launch_noalloc<MaxI32>(in, out, n, ws, stream);
    else
        e = launch_noalloc<XorU32>(in, out, n, ws, stream);
    return e == cudaSuccess ? DEVSCAN_OK : DEVSCAN_ERR_CUDA;
}
