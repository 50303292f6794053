/*
 * devscan -- device-wide parallel prefix scan, stream compaction and radix
 * one-bit split for one NVIDIA GB300 GPU (sm_103a).
 *
 * C ABI.  Every pointer argument of a compute call is a DEVICE pointer owned
 * by the caller; the library never frees, retains or reallocates it.  Every
 * compute call is asynchronous and ordered on the caller's `stream`: it
 * validates its arguments on the host, launches its kernels and returns.
 * Launch errors are returned immediately as DEVSCAN_ERR_CUDA; errors raised
 * inside a kernel (a bounded inter-block wait that ran out) are recorded in a
 * per-stream device word and reported by devscan_device_status().
 *
 * Scratch memory.  The single-pass kernels keep a small per-stream workspace
 * (one 8-byte status word per tile of the largest input seen, plus a few
 * counters) that the library allocates stream-ordered on first use
 * (cudaMallocAsync) and reuses for later calls on the same stream.  Calls on
 * one stream never race on it; calls on different streams use different
 * workspaces.  devscan_stream_release() frees a stream's workspace.
 *
 * Pages the operations follow:
 *   [P1] geek-doc.cn/chip-design/intermediate/parallel-prefix-scan,
 *        "并行前缀和 scan: Hillis-Steele、Blelloch 与 warp shuffle 三种写法";
 *   [P2] lpnh.cn/news/2866224, "并行扫描 Scan/Prefix Sum";
 *   [P3] pgsm.cn/news/414823, "SIMT数据依赖与并行前缀和：从原理到流压缩实战".
 */
#ifndef DEVSCAN_H
#define DEVSCAN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Associative operators (P1 section 三 and P2 section 3.3: any associative
 * operator can be scanned).  ADD wraps modulo 2^32 on the integer types;
 * MAX compares as signed for int32 and unsigned for uint32, and follows
 * fmaxf for fp32; XOR is defined on the integer types only. */
typedef enum devscan_op {
    DEVSCAN_OP_ADD = 0,
    DEVSCAN_OP_MAX = 1,
    DEVSCAN_OP_XOR = 2
} devscan_op;

typedef enum devscan_status {
    DEVSCAN_OK = 0,
    DEVSCAN_ERR_INVALID = 1,     /* bad argument: null pointer with n > 0, bad
                                    bit index, overlapping buffers, size limit */
    DEVSCAN_ERR_UNSUPPORTED = 2, /* operator not defined for the type (xor on fp32) */
    DEVSCAN_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    DEVSCAN_ERR_TIMEOUT = 4,     /* an inter-block wait gave up (device side) */
    DEVSCAN_ERR_NOMEM = 5        /* the workspace could not be allocated */
} devscan_status;

/* ---------------------------------------------------------------------------
 * Scans.  P1 section 一: inclusive y[i] = x[0] ⊕ ... ⊕ x[i]; exclusive
 * z[i] = x[0] ⊕ ... ⊕ x[i-1] with z[0] the identity of ⊕ (0 for add and
 * xor, INT32_MIN for int32 max, 0 for uint32 max, -inf for fp32 max).
 *
 *   in, out : device arrays of n elements.  out == in (in place) is allowed;
 *             any other overlap is not checked and gives undefined results.
 *             16-byte aligned pointers take the vectorised path, any other
 *             element-aligned pointers are accepted on a scalar path.
 *   n       : element count; n == 0 is a no-op returning DEVSCAN_OK.
 *   op      : DEVSCAN_OP_*; XOR on fp32 returns DEVSCAN_ERR_UNSUPPORTED.
 *   stream  : the CUDA stream to order the work on (0 = legacy default).
 *
 * fp32 add is computed in fp32 in a parallel order; its result differs from
 * a serial fp64 sum by at most a small multiple of fp32 rounding of the
 * running sum of |x| (P1 pitfalls: floating-point addition is not
 * associative), and may differ between runs in the last bits.
 * ------------------------------------------------------------------------- */
devscan_status scan_inclusive_i32(const int32_t *in, int32_t *out, size_t n,
                                  devscan_op op, cudaStream_t stream);
devscan_status scan_inclusive_u32(const uint32_t *in, uint32_t *out, size_t n,
                                  devscan_op op, cudaStream_t stream);
devscan_status scan_inclusive_f32(const float *in, float *out, size_t n,
                                  devscan_op op, cudaStream_t stream);
devscan_status scan_exclusive_i32(const int32_t *in, int32_t *out, size_t n,
                                  devscan_op op, cudaStream_t stream);
devscan_status scan_exclusive_u32(const uint32_t *in, uint32_t *out, size_t n,
                                  devscan_op op, cudaStream_t stream);
devscan_status scan_exclusive_f32(const float *in, float *out, size_t n,
                                  devscan_op op, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Scans of host arrays: the host-side entry to the scans above, for callers
 * whose data lives in host memory (P2 section 5.3: the copies and the scan
 * are ordered on a CUDA stream, so work on two streams overlaps one's
 * transfers with the other's; the scan itself is P1 section 一).  In order on
 * `stream`:
 *   1. h_in[0 .. n) is copied into d_in (host to device);
 *   2. d_in is scanned into d_out by the device scan above (same operators,
 *      identities, paths and accuracy);
 *   3. d_out is copied into h_out[0 .. n) (device to host).
 * The call returns once the three steps are queued; h_out holds the result
 * when the stream has reached this point (synchronise the stream, or record
 * an event after the call).
 *
 *   h_in, h_out : host arrays of n elements; they may be the same array.
 *                 Page-locked (pinned) memory makes the copies asynchronous;
 *                 with pageable memory CUDA stages them and they are slower.
 *                 The caller keeps both valid and untouched until the
 *                 stream has reached this point.
 *   d_in, d_out : device arrays of n elements owned by the caller (the call
 *                 allocates no array of n elements); d_out may equal d_in;
 *                 otherwise they must not overlap (DEVSCAN_ERR_INVALID).
 *                 16-byte aligned buffers take the vectorised paths.
 * Other arguments and errors as the scans; a failed copy returns
 * DEVSCAN_ERR_CUDA.  Traffic: n * sizeof(T) bytes over the host link in each
 * direction, plus the scan's 2 * n * sizeof(T) bytes of device memory.
 * Calls on two streams overlap one call's download with the other's upload.
 * ------------------------------------------------------------------------- */
devscan_status scan_inclusive_host_i32(const int32_t *h_in, int32_t *h_out, size_t n, devscan_op op,
                                       int32_t *d_in, int32_t *d_out, cudaStream_t stream);
devscan_status scan_inclusive_host_u32(const uint32_t *h_in, uint32_t *h_out, size_t n, devscan_op op,
                                       uint32_t *d_in, uint32_t *d_out, cudaStream_t stream);
devscan_status scan_inclusive_host_f32(const float *h_in, float *h_out, size_t n, devscan_op op,
                                       float *d_in, float *d_out, cudaStream_t stream);
devscan_status scan_exclusive_host_i32(const int32_t *h_in, int32_t *h_out, size_t n, devscan_op op,
                                       int32_t *d_in, int32_t *d_out, cudaStream_t stream);
devscan_status scan_exclusive_host_u32(const uint32_t *h_in, uint32_t *h_out, size_t n, devscan_op op,
                                       uint32_t *d_in, uint32_t *d_out, cudaStream_t stream);
devscan_status scan_exclusive_host_f32(const float *h_in, float *h_out, size_t n, devscan_op op,
                                       float *d_in, float *d_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Scans with a carry-in, and the fold of an array: the pieces of a scan whose
 * input is split into contiguous shards, one per device (P1 section 四 and
 * P2 section 3.2: reduce each part, scan the part totals, give every part
 * its offset -- here the parts are shards instead of blocks).  Shard r of P:
 *   1. reduce_T(shard_r, n_r, op, &total_r)      its own total;
 *   2. the P totals are exchanged (an all-gather of P scalars, outside this
 *      library: each device keeps the array totals[0 .. P) in its memory);
 *   3. reduce_T(totals, r, op, &carry_r)         the fold of the earlier
 *      shards' totals (the identity for r == 0);
 *   4. scan_*_carry_T(shard_r, out_r, n_r, op, &carry_r)   its scan.
 * The concatenated out_r then equal the scan of the whole array.
 *
 * scan_{inclusive,exclusive}_carry_T: the scans above with
 *   out[i] = carry ⊕ (scan of in)[i], carry = *carry_in,
 * i.e. the scan of the array that carry_in's value would precede; exclusive
 * out[0] is the carry itself.
 *   carry_in : device pointer to one T, 4-byte aligned, read on the stream
 *              (so it may be written by earlier work on the same stream); it
 *              must not overlap out (DEVSCAN_ERR_INVALID); NULL means the
 *              identity (the plain scan).
 * Other arguments, paths, limits and errors as the scans above.  fp32 add
 * adds the carry in fp32 (one more rounding per element).
 *
 * reduce_T: *total = in[0] ⊕ in[1] ⊕ ... ⊕ in[n-1], the identity of ⊕ when
 * n == 0.  One read of the input (4 bytes per element), one launch; fp32
 * add is folded in a fixed order (the same n and alignment give the same
 * bits).  in: device T[n], 4-byte aligned (NULL allowed when n == 0);
 * total: device T, 4-byte aligned, not inside in.  Operators and errors as
 * the scans.
 * ------------------------------------------------------------------------- */
devscan_status scan_inclusive_carry_i32(const int32_t *in, int32_t *out, size_t n, devscan_op op,
                                        const int32_t *carry_in, cudaStream_t stream);
devscan_status scan_inclusive_carry_u32(const uint32_t *in, uint32_t *out, size_t n, devscan_op op,
                                        const uint32_t *carry_in, cudaStream_t stream);
devscan_status scan_inclusive_carry_f32(const float *in, float *out, size_t n, devscan_op op,
                                        const float *carry_in, cudaStream_t stream);
devscan_status scan_exclusive_carry_i32(const int32_t *in, int32_t *out, size_t n, devscan_op op,
                                        const int32_t *carry_in, cudaStream_t stream);
devscan_status scan_exclusive_carry_u32(const uint32_t *in, uint32_t *out, size_t n, devscan_op op,
                                        const uint32_t *carry_in, cudaStream_t stream);
devscan_status scan_exclusive_carry_f32(const float *in, float *out, size_t n, devscan_op op,
                                        const float *carry_in, cudaStream_t stream);
devscan_status reduce_i32(const int32_t *in, size_t n, devscan_op op, int32_t *total, cudaStream_t stream);
devscan_status reduce_u32(const uint32_t *in, size_t n, devscan_op op, uint32_t *total, cudaStream_t stream);
devscan_status reduce_f32(const float *in, size_t n, devscan_op op, float *total, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Segmented scans (P2 section 7.2 names the segmented scan for sparse data):
 * heads[i] != 0 starts a new segment at i (element 0 always starts one) and
 * every segment is scanned on its own, the running value returning to the
 * operator's identity at each segment start:
 *   inclusive  out[i] = in[s] (+) ... (+) in[i],
 *   exclusive  out[i] = identity (+) in[s] (+) ... (+) in[i-1],
 * with s the start of i's segment (exclusive: identity at every start).
 *
 *   in, out : device T[n], 4-byte aligned; out may equal in (in place),
 *             otherwise the two must not overlap;
 *   heads   : device uint8[n], nonzero = segment start; must not overlap out.
 * Operators, identities, fp32 accuracy (per segment: |err_i| within
 * 1e-5 * sum of |in[j]| over i's segment up to i), limits and errors as the
 * scans above.  Traffic: 5 bytes read and 4 written per element.
 * ------------------------------------------------------------------------- */
devscan_status segmented_scan_inclusive_i32(const int32_t *in, const uint8_t *heads, int32_t *out,
                                            size_t n, devscan_op op, cudaStream_t stream);
devscan_status segmented_scan_inclusive_u32(const uint32_t *in, const uint8_t *heads, uint32_t *out,
                                            size_t n, devscan_op op, cudaStream_t stream);
devscan_status segmented_scan_inclusive_f32(const float *in, const uint8_t *heads, float *out,
                                            size_t n, devscan_op op, cudaStream_t stream);
devscan_status segmented_scan_exclusive_i32(const int32_t *in, const uint8_t *heads, int32_t *out,
                                            size_t n, devscan_op op, cudaStream_t stream);
devscan_status segmented_scan_exclusive_u32(const uint32_t *in, const uint8_t *heads, uint32_t *out,
                                            size_t n, devscan_op op, cudaStream_t stream);
devscan_status segmented_scan_exclusive_f32(const float *in, const uint8_t *heads, float *out,
                                            size_t n, devscan_op op, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Stream compaction (P1 section 一; P2 section 4.1; P3 sections 4.1-4.2):
 * out[0 .. *count) receives, in input order, every in[i] whose flags[i] is
 * nonzero; *count is the number kept.  Each kept element's slot is the
 * exclusive add-scan of the 0/1 predicate, computed on the device.
 *
 *   in     : device int32[n];  flags : device uint8[n] (nonzero = keep);
 *   out    : device int32 with room for n elements (only *count are written);
 *   count  : device int32, written with the number kept (0 when n == 0).
 *   n      : at most INT32_MAX, else DEVSCAN_ERR_INVALID.
 *   out must not overlap in or flags (DEVSCAN_ERR_INVALID).
 * From 2^23 elements (in and flags 16-byte aligned) it runs in two launches:
 * a count of every 512-element part (keep mask, count, offset), then a warp
 * per part writing its kept values; 18 words per 512 elements of per-stream
 * scratch are allocated stream-ordered on first use (DEVSCAN_ERR_NOMEM if
 * that fails).  Smaller or unaligned inputs take a single-pass kernel.
 * ------------------------------------------------------------------------- */
devscan_status compact_i32(const int32_t *in, const uint8_t *flags, int32_t *out,
                           int32_t *count, size_t n, cudaStream_t stream);

/* Stream compaction with the predicate evaluated on the device (P3 section
 * 3.3: each element contributes 1 when it is to be output, 0 otherwise; P2
 * section 4.1, the predicate applied element by element): out[0 .. *count)
 * receives, in input order, every in[i] with in[i] > threshold (signed
 * compare).  No flag array is read, so the traffic is 4 bytes per element
 * plus 4 per kept element.  Arguments, limits and errors as compact_i32,
 * without flags.
 * From 2^19 elements (in 16-byte aligned) the call is one cooperative launch
 * (one block per SM): it first reads the values once and keeps the kept ones
 * in shared memory, which succeeds while they fit (at 2^26 elements, up to
 * about 10% kept), and otherwise goes on as a pipeline that reads them again.
 * After a capture gives up, the stream skips it for its next 16 calls.  That
 * state lives in the stream's workspace and affects only how the work is
 * done, never the result.
 * Smaller or unaligned inputs take a single-pass kernel. */
devscan_status compact_gt_i32(const int32_t *in, int32_t threshold, int32_t *out,
                              int32_t *count, size_t n, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Bracket check fused into the scan (P1 section 一: '(' counts +1 and ')'
 * -1; a negative running sum means a surplus ')', a nonzero final sum means
 * the brackets do not pair up, and one scan answers both).  One pass over
 * in[0 .. n):
 *   out       : the inclusive int32 add-scan (wrapping modulo 2^32), or NULL
 *               to skip storing it (the check alone then only reads in);
 *               may equal in; 4-byte aligned;
 *   result[0] : 1 if some inclusive prefix is negative (as int32), else 0;
 *   result[1] : the final inclusive prefix (0 when n == 0).
 * result is a device int32[2], 4-byte aligned, overlapping neither in nor
 * out (else DEVSCAN_ERR_INVALID); it is cleared on the stream first.  The
 * brackets are balanced iff result[0] == 0 and result[1] == 0.  Any int32
 * weights are accepted; the answers refer to the wrapped int32 prefixes.
 * n limits and errors as the scans.
 * ------------------------------------------------------------------------- */
devscan_status bracket_scan_i32(const int32_t *in, int32_t *out, int32_t *result, size_t n,
                                cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Radix-sort one-bit split (P1 section 一, radix sort; P2 section 4.2): a
 * stable partition of keys by bit `bit`.  With zerosBefore(i) the exclusive
 * add-scan of (bit is 0) and Z the total number of zeros, a key whose bit is
 * 0 goes to out[zerosBefore(i)] and a key whose bit is 1 goes to
 * out[Z + i - zerosBefore(i)].
 *
 *   keys, out : device uint32[n], not overlapping (DEVSCAN_ERR_INVALID);
 *   bit       : 0..31, else DEVSCAN_ERR_INVALID;
 *   n         : at most INT32_MAX, else DEVSCAN_ERR_INVALID.
 * From 2^20 keys (keys 16-byte aligned): a launch counting every 1,024-key
 * part's zeros into part offsets and Z, then a warp per part writing its two
 * runs; one word per 1,024 keys of per-stream scratch is allocated
 * stream-ordered on first use (DEVSCAN_ERR_NOMEM if that fails).  Below, a
 * zero-count pass, then the single-pass split.
 * ------------------------------------------------------------------------- */
devscan_status split_bit_u32(const uint32_t *keys, uint32_t *out, int bit, size_t n,
                             cudaStream_t stream);

/* Least-significant-bit-first radix sort of uint32 keys by 32 one-bit splits
 * (P1 section 一: one bit per round; each round's core is a scan).  Pass b
 * counts the zeros of bit b+1 while it scatters, and one count pass runs
 * before pass 0.  From 2^20 keys (keys and tmp 16-byte aligned) each pass
 * is the two-launch split, whose write launch counts bit b+1's zeros per
 * 1,024-key part of its output, plus a small launch turning those counts into
 * the next pass's offsets; 2 words per 1,024 keys of per-stream scratch are
 * allocated stream-ordered on first use (DEVSCAN_ERR_NOMEM if that fails).
 * Otherwise each pass is the pipelined (or one-tile) split, which needs only
 * the total zero count of bit b+1.
 *
 *   keys : device uint32[n]; sorted ascending in place on return (stream order);
 *   tmp  : device uint32[n] scratch owned by the caller, not overlapping keys;
 *   n    : at most INT32_MAX, else DEVSCAN_ERR_INVALID.
 * ------------------------------------------------------------------------- */
devscan_status radix_sort_u32(uint32_t *keys, uint32_t *tmp, size_t n, cudaStream_t stream);

/* LSD radix sort of uint32 keys by 8-bit digits: 4 passes (P1 section 一:
 * a round may take "one or several bits"; P2 section 4.2: per-digit counts,
 * a prefix over them, then the scatter).  Each pass counts the 256 digit
 * values of every 8,192-key tile, scans the digit-major count array with the
 * library's exclusive add-scan (giving every (digit, tile) run its output
 * position), and scatters each tile's keys stably as one contiguous run per
 * digit.  Same arguments and result as radix_sort_u32 (the result is in
 * keys; n at most INT32_MAX); a per-stream scratch of n / 32 words holds the
 * counts (allocated stream-ordered on first use). */
devscan_status radix_sort_digits_u32(uint32_t *keys, uint32_t *tmp, size_t n, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Status and housekeeping.
 * ------------------------------------------------------------------------- */

/* Synchronises `stream`, then reports and clears the device-side error word
 * of the stream's workspace: DEVSCAN_ERR_TIMEOUT if a bounded inter-block
 * wait gave up since the last query (the affected results are not valid;
 * the workspace is reset so that later calls start clean),
 * DEVSCAN_ERR_CUDA if the synchronisation failed, else DEVSCAN_OK. */
devscan_status devscan_device_status(cudaStream_t stream);

/* Static English text for a status code. */
const char *devscan_status_string(devscan_status status);

/* Frees the workspace tied to `stream` (stream-ordered, so work already
 * queued on it finishes first).  Call before destroying a stream that ran
 * devscan work; a later call on the stream allocates a new workspace. */
devscan_status devscan_stream_release(cudaStream_t stream);

/* Self-test of the bounded inter-block wait: launches two blocks on
 * `stream` where the second waits for a tile status that nothing ever
 * publishes, giving up after `spin_limit` polls.  Afterwards
 * devscan_device_status(stream) returns DEVSCAN_ERR_TIMEOUT.  No kernel
 * faults or hangs. */
devscan_status devscan_selftest_stalled_wait(unsigned int spin_limit, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Allocation-free int32 exclusive scan.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory -- code
 * whose GPU memory is owned by another allocator (a framework's caching
 * pool that has reserved the device, where an extra cudaMalloc can fail or
 * force the pool to give memory back) and code that must not allocate after
 * start-up (latency-critical or certified paths).  The other entry points
 * allocate their per-stream workspace on first use; this one never calls
 * cudaMalloc, cudaMallocAsync, cudaFree or any allocating routine.
 *
 * Same semantics and arguments as scan_exclusive_i32 (DEVSCAN_OP_ADD, MAX or
 * XOR; in == out allowed).  Its scratch -- the tile status words of the
 * single-pass look-back and a few counters -- is one fixed array compiled
 * into the library (static device memory, 528 KiB + 256 B on every GPU that
 * loads the library, held until the process exits):
 *   - n > DEVSCAN_NOALLOC_MAX_N returns DEVSCAN_ERR_INVALID (nothing runs);
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture;
 *   - every call shares the one array: calls that may overlap on the GPU
 *     (different streams without ordering between them) race and give wrong
 *     results; calls on one stream are safe.  Each call clears the tile
 *     counter it needs at zero; stale status words of earlier calls are
 *     ignored through their epoch tag.
 *   - a device-side wait that runs out (never seen in normal operation) is
 *     not reported by this entry point.
 * ------------------------------------------------------------------------- */
#define DEVSCAN_NOALLOC_MAX_N ((size_t)1 << 28)

devscan_status scan_exclusive_i32_noalloc(const int32_t *in, int32_t *out, size_t n,
                                          devscan_op op, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DEVSCAN_H */
