"""devscan for GB300: device-wide prefix scan, stream compaction and the
radix one-bit split as hand-written sm_103a CUDA kernels behind a C ABI.

The functions below take CUDA tensors (PyTorch is used for device memory
and streams only), pass their device pointers and the current CUDA stream
to ``libdevscan.so`` and return.  All work is asynchronous on that stream.
``scan_host`` is the host-buffer entry: the library copies a pinned host
array to the device, scans it and copies the result back.
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import DevscanError, OPS, load

__all__ = ["scan_inclusive", "scan_exclusive", "scan_inclusive_carry", "scan_exclusive_carry", "reduce",
           "sharded_scan", "exchange_totals", "compact", "split_bit", "radix_sort", "radix_sort_digits", "scan_host",
           "compact_greater", "bracket_scan", "segmented_scan_inclusive", "segmented_scan_exclusive",
           "device_status", "set_carry_mode", "stream_release", "selftest_stalled_wait", "DevscanError",
           "load"]

_SUFFIX = {torch.int32: "i32", torch.float32: "f32"}
if hasattr(torch, "uint32"):
    _SUFFIX[torch.uint32] = "u32"


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check_cuda(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _scan(direction: str, x: torch.Tensor, out, op: str, stream, dtype_override=None):
    _check_cuda(x, "x")
    suffix = dtype_override or _SUFFIX.get(x.dtype)
    if suffix is None:
        raise TypeError(f"unsupported dtype {x.dtype} (int32, uint32, float32)")
    if out is None:
        out = torch.empty_like(x)
    _check_cuda(out, "out")
    if out.numel() != x.numel() or out.dtype != x.dtype:
        raise ValueError("out must match x in size and dtype")
    fn = getattr(load(), f"scan_{direction}_{suffix}")
    _lib.check(fn(x.data_ptr(), out.data_ptr(), x.numel(), OPS[op], _stream_handle(stream)),
               f"scan_{direction}_{suffix}")
    return out


def scan_inclusive(x: torch.Tensor, out: torch.Tensor | None = None, op: str = "add", stream=None,
                   as_uint32: bool = False) -> torch.Tensor:
    """y[i] = x[0] op ... op x[i].  ``as_uint32`` treats an int32 tensor's
    bits as uint32 (unsigned max)."""
    return _scan("inclusive", x, out, op, stream, "u32" if as_uint32 else None)


def scan_exclusive(x: torch.Tensor, out: torch.Tensor | None = None, op: str = "add", stream=None,
                   as_uint32: bool = False) -> torch.Tensor:
    """z[i] = x[0] op ... op x[i-1]; z[0] = identity of op."""
    return _scan("exclusive", x, out, op, stream, "u32" if as_uint32 else None)


def _carry_scan(direction: str, x: torch.Tensor, carry: torch.Tensor | None, out, op: str, stream,
                dtype_override=None):
    _check_cuda(x, "x")
    suffix = dtype_override or _SUFFIX.get(x.dtype)
    if suffix is None:
        raise TypeError(f"unsupported dtype {x.dtype} (int32, uint32, float32)")
    if carry is not None:
        _check_cuda(carry, "carry")
        if carry.dtype != x.dtype or carry.numel() < 1:
            raise ValueError("carry must be a device tensor of x's dtype holding one element")
    if out is None:
        out = torch.empty_like(x)
    _check_cuda(out, "out")
    if out.numel() != x.numel() or out.dtype != x.dtype:
        raise ValueError("out must match x in size and dtype")
    name = f"scan_{direction}_carry_{suffix}"
    _lib.check(getattr(load(), name)(x.data_ptr(), out.data_ptr(), x.numel(), OPS[op],
                                     None if carry is None else carry.data_ptr(), _stream_handle(stream)), name)
    return out


def scan_inclusive_carry(x: torch.Tensor, carry: torch.Tensor | None, out: torch.Tensor | None = None,
                         op: str = "add", stream=None, as_uint32: bool = False) -> torch.Tensor:
    """y[i] = carry op x[0] op ... op x[i], ``carry`` a one-element device
    tensor (None: the identity)."""
    return _carry_scan("inclusive", x, carry, out, op, stream, "u32" if as_uint32 else None)


def scan_exclusive_carry(x: torch.Tensor, carry: torch.Tensor | None, out: torch.Tensor | None = None,
                         op: str = "add", stream=None, as_uint32: bool = False) -> torch.Tensor:
    """z[i] = carry op x[0] op ... op x[i-1]; z[0] = carry."""
    return _carry_scan("exclusive", x, carry, out, op, stream, "u32" if as_uint32 else None)


def reduce(x: torch.Tensor, op: str = "add", out: torch.Tensor | None = None, stream=None,
           as_uint32: bool = False) -> torch.Tensor:
    """Fold of all of ``x`` under ``op`` into a one-element device tensor
    (the identity for an empty ``x``)."""
    _check_cuda(x, "x")
    suffix = "u32" if as_uint32 else _SUFFIX.get(x.dtype)
    if suffix is None:
        raise TypeError(f"unsupported dtype {x.dtype} (int32, uint32, float32)")
    if out is None:
        out = torch.empty(1, dtype=x.dtype, device=x.device)
    _check_cuda(out, "out")
    if out.dtype != x.dtype or out.numel() < 1:
        raise ValueError("out must hold one element of x's dtype")
    name = f"reduce_{suffix}"
    _lib.check(getattr(load(), name)(x.data_ptr() if x.numel() else None, x.numel(), OPS[op], out.data_ptr(),
                                     _stream_handle(stream)), name)
    return out


def exchange_totals(total: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of one total per rank: returns a tensor of ``world_size``
    elements on ``total``'s device, element r from rank r (the one exchange
    step of a sharded scan; NCCL for device tensors, gloo for host
    tensors).  A single process returns ``total`` itself."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return total.reshape(1)
    world = dist.get_world_size(group)
    totals = torch.empty(world, dtype=total.dtype, device=total.device)
    dist.all_gather_into_tensor(totals, total.reshape(1).contiguous(), group=group)
    return totals


def sharded_scan(shard: torch.Tensor, out: torch.Tensor | None = None, inclusive: bool = False, op: str = "add",
                 group=None, stream=None, as_uint32: bool = False) -> torch.Tensor:
    """This rank's part of the scan of an array split into contiguous shards,
    shard r on rank r of ``group`` (in rank order).  The library folds this
    shard's total, the ranks exchange their totals (one all-gather of one
    element each), the library folds the totals of the ranks before this
    one into a carry and scans the shard from it.  Every rank calls it; the
    ranks' outputs, concatenated in rank order, are the scan of the whole
    array."""
    import torch.distributed as dist
    rank = dist.get_rank(group) if dist.is_available() and dist.is_initialized() else 0
    total = reduce(shard, op, stream=stream, as_uint32=as_uint32)
    totals = exchange_totals(total, group)
    carry = reduce(totals[:rank], op, stream=stream, as_uint32=as_uint32)
    fn = scan_inclusive_carry if inclusive else scan_exclusive_carry
    return fn(shard, carry, out, op=op, stream=stream, as_uint32=as_uint32)


def sharded_compact(values: torch.Tensor, flags: torch.Tensor | None = None, threshold: int | None = None,
                    out: torch.Tensor | None = None, group=None, stream=None):
    """This rank's part of the order-preserving compaction of an array split
    into contiguous shards, shard r on rank r of ``group`` (in rank order).
    The library compacts the shard (the values whose flag is nonzero, or the
    values greater than ``threshold``), the ranks exchange their kept counts
    (one all-gather of one count each), and the library folds the counts of
    the ranks before this one into this rank's output offset and all of them
    into the total.  Returns (out, count, offset, total), all on the device:
    the first ``count`` elements of ``out`` are this rank's kept values,
    elements offset .. offset + count - 1 of the whole compaction."""
    import torch.distributed as dist
    if (flags is None) == (threshold is None):
        raise ValueError("give either flags or a threshold")
    rank = dist.get_rank(group) if dist.is_available() and dist.is_initialized() else 0
    if threshold is None:
        out, count = compact(values, flags, out, stream=stream)
    else:
        out, count = compact_greater(values, threshold, out, stream=stream)
    counts = exchange_totals(count, group)
    offset = reduce(counts[:rank], "add", stream=stream)
    total = reduce(counts, "add", stream=stream)
    return out, count, offset, total


def _segscan(direction: str, x: torch.Tensor, heads: torch.Tensor, out, op: str, stream, dtype_override=None):
    _check_cuda(x, "x")
    _check_cuda(heads, "heads")
    suffix = dtype_override or _SUFFIX.get(x.dtype)
    if suffix is None:
        raise TypeError(f"unsupported dtype {x.dtype} (int32, uint32, float32)")
    if heads.dtype != torch.uint8 or heads.numel() != x.numel():
        raise ValueError("heads must be a uint8 tensor of x's length")
    if out is None:
        out = torch.empty_like(x)
    _check_cuda(out, "out")
    if out.numel() != x.numel() or out.dtype != x.dtype:
        raise ValueError("out must match x in size and dtype")
    name = f"segmented_scan_{direction}_{suffix}"
    _lib.check(getattr(load(), name)(x.data_ptr(), heads.data_ptr(), out.data_ptr(), x.numel(), OPS[op],
                                     _stream_handle(stream)), name)
    return out


def segmented_scan_inclusive(x: torch.Tensor, heads: torch.Tensor, out: torch.Tensor | None = None,
                             op: str = "add", stream=None, as_uint32: bool = False) -> torch.Tensor:
    """Inclusive scan restarted at every nonzero ``heads[i]`` (element 0
    always starts a segment)."""
    return _segscan("inclusive", x, heads, out, op, stream, "u32" if as_uint32 else None)


def segmented_scan_exclusive(x: torch.Tensor, heads: torch.Tensor, out: torch.Tensor | None = None,
                             op: str = "add", stream=None, as_uint32: bool = False) -> torch.Tensor:
    """Exclusive scan restarted at every nonzero ``heads[i]``: the identity
    at each segment start."""
    return _segscan("exclusive", x, heads, out, op, stream, "u32" if as_uint32 else None)


def compact(values: torch.Tensor, flags: torch.Tensor, out: torch.Tensor | None = None,
            count: torch.Tensor | None = None, stream=None):
    """Order-preserving compaction.  Returns (out, count): the first
    ``count`` elements of ``out`` are the values whose flag is nonzero.
    Both stay on the device; nothing synchronises."""
    _check_cuda(values, "values")
    _check_cuda(flags, "flags")
    if values.dtype != torch.int32 or flags.dtype != torch.uint8:
        raise TypeError("values must be int32 and flags uint8")
    if values.numel() != flags.numel():
        raise ValueError("values and flags differ in length")
    if out is None:
        out = torch.empty_like(values)
    if count is None:
        count = torch.empty(1, dtype=torch.int32, device=values.device)
    _check_cuda(out, "out")
    _check_cuda(count, "count")
    _lib.check(load().compact_i32(values.data_ptr(), flags.data_ptr(), out.data_ptr(), count.data_ptr(),
                                  values.numel(), _stream_handle(stream)), "compact_i32")
    return out, count


def compact_greater(values: torch.Tensor, threshold: int, out: torch.Tensor | None = None,
                    count: torch.Tensor | None = None, stream=None):
    """Order-preserving compaction of the int32 values greater than
    ``threshold`` (signed), the predicate evaluated on the device.  Returns
    (out, count) as :func:`compact`."""
    _check_cuda(values, "values")
    if values.dtype != torch.int32:
        raise TypeError("values must be int32")
    if out is None:
        out = torch.empty_like(values)
    if count is None:
        count = torch.empty(1, dtype=torch.int32, device=values.device)
    _check_cuda(out, "out")
    _check_cuda(count, "count")
    _lib.check(load().compact_gt_i32(values.data_ptr(), int(threshold), out.data_ptr(), count.data_ptr(),
                                     values.numel(), _stream_handle(stream)), "compact_gt_i32")
    return out, count


def bracket_scan(weights: torch.Tensor, out: torch.Tensor | None = None, result: torch.Tensor | None = None,
                 store: bool = True, stream=None):
    """Inclusive int32 add-scan of +1/-1 bracket weights with the bracket
    check in the same pass.  Returns (out or None, result): result[0] is 1
    when some running sum is negative, result[1] the final sum.  With
    ``store=False`` the scan is not written (the check alone)."""
    _check_cuda(weights, "weights")
    if weights.dtype != torch.int32:
        raise TypeError("weights must be int32")
    if store and out is None:
        out = torch.empty_like(weights)
    if not store:
        out = None
    if result is None:
        result = torch.empty(2, dtype=torch.int32, device=weights.device)
    _check_cuda(result, "result")
    if out is not None:
        _check_cuda(out, "out")
    _lib.check(load().bracket_scan_i32(weights.data_ptr(), None if out is None else out.data_ptr(),
                                       result.data_ptr(), weights.numel(), _stream_handle(stream)),
               "bracket_scan_i32")
    return out, result


def split_bit(keys: torch.Tensor, bit: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Stable partition of 32-bit keys by bit ``bit``: zeros first."""
    _check_cuda(keys, "keys")
    if keys.element_size() != 4 or keys.is_floating_point():
        raise TypeError("keys must be a 32-bit integer tensor (bits read as uint32)")
    if out is None:
        out = torch.empty_like(keys)
    _check_cuda(out, "out")
    _lib.check(load().split_bit_u32(keys.data_ptr(), out.data_ptr(), int(bit), keys.numel(),
                                    _stream_handle(stream)), "split_bit_u32")
    return out


def radix_sort(keys: torch.Tensor, tmp: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """In-place ascending sort of 32-bit keys (bits read as uint32) by 32
    one-bit splits; ``tmp`` is a same-size scratch tensor."""
    _check_cuda(keys, "keys")
    if keys.element_size() != 4 or keys.is_floating_point():
        raise TypeError("keys must be a 32-bit integer tensor (bits read as uint32)")
    if tmp is None:
        tmp = torch.empty_like(keys)
    _check_cuda(tmp, "tmp")
    _lib.check(load().radix_sort_u32(keys.data_ptr(), tmp.data_ptr(), keys.numel(), _stream_handle(stream)),
               "radix_sort_u32")
    return keys


def radix_sort_digits(keys: torch.Tensor, tmp: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """In-place ascending sort of 32-bit keys (bits read as uint32) by 4
    passes of 8-bit digits; ``tmp`` is a same-size scratch tensor."""
    _check_cuda(keys, "keys")
    if keys.element_size() != 4 or keys.is_floating_point():
        raise TypeError("keys must be a 32-bit integer tensor (bits read as uint32)")
    if tmp is None:
        tmp = torch.empty_like(keys)
    _check_cuda(tmp, "tmp")
    _lib.check(load().radix_sort_digits_u32(keys.data_ptr(), tmp.data_ptr(), keys.numel(),
                                            _stream_handle(stream)), "radix_sort_digits_u32")
    return keys


def scan_host(x_host: torch.Tensor, inclusive: bool = False, op: str = "add", device="cuda",
              stream=None, out_host: torch.Tensor | None = None, work=None,
              synchronize: bool = True, as_uint32: bool = False) -> torch.Tensor:
    """Scan a host array end to end through the library's host entry
    (``scan_{inclusive,exclusive}_host_T``): host-to-device copy, device
    scan, device-to-host copy, all queued by the library on ``stream``.
    Pinned host tensors make the copies asynchronous.  ``work`` may pass
    preallocated (device input, device output) tensors.  With
    ``synchronize`` (the default) it returns once the result is in
    ``out_host``; without, it returns at once and the result is there when
    ``stream`` has reached this point, so calls on two streams overlap one
    call's download with the next one's upload."""
    if x_host.is_cuda:
        raise ValueError("x_host must be a host tensor")
    if not x_host.is_contiguous():
        raise ValueError("x_host must be contiguous")
    suffix = "u32" if as_uint32 else _SUFFIX.get(x_host.dtype)
    if suffix is None:
        raise TypeError(f"unsupported dtype {x_host.dtype} (int32, uint32, float32)")
    s = stream if stream is not None else torch.cuda.current_stream()
    if work is None:
        d_in = torch.empty(x_host.shape, dtype=x_host.dtype, device=device)
        d_out = torch.empty_like(d_in)
    else:
        d_in, d_out = work
        _check_cuda(d_in, "work[0]")
        _check_cuda(d_out, "work[1]")
        if d_in.numel() < x_host.numel() or d_out.numel() < x_host.numel():
            raise ValueError("work tensors are smaller than x_host")
    if out_host is None:
        out_host = torch.empty(x_host.shape, dtype=x_host.dtype, pin_memory=x_host.is_pinned())
    if out_host.is_cuda or out_host.numel() != x_host.numel() or out_host.dtype != x_host.dtype:
        raise ValueError("out_host must be a host tensor matching x_host")
    name = f"scan_{'inclusive' if inclusive else 'exclusive'}_host_{suffix}"
    _lib.check(getattr(load(), name)(x_host.data_ptr(), out_host.data_ptr(), x_host.numel(), OPS[op],
                                     d_in.data_ptr(), d_out.data_ptr(), _stream_handle(s)), name)
    if synchronize:
        s.synchronize()
    return out_host


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) its device-side status."""
    return load().devscan_device_status(_stream_handle(stream))


def set_carry_mode(mode: str) -> None:
    """Measurement hook (``devscan_measure_set_carry_mode``): 'default',
    'lookback' (one tile per block), 'rts' (reduce-then-scan), 'pipelined'
    (persistent warp-specialised single pass) or 'l2' (the cooperative forms:
    the L2-resident scan, the one-read bracket check, the two-launch
    compaction with flags and split).  Applies to the calling thread's later
    calls only."""
    code = {"default": 0, "lookback": 1, "rts": 2, "pipelined": 3, "l2": 4}[mode]
    _lib.check(load().devscan_measure_set_carry_mode(code), "devscan_measure_set_carry_mode")


def stream_release(stream=None) -> None:
    _lib.check(load().devscan_stream_release(_stream_handle(stream)), "devscan_stream_release")


def selftest_stalled_wait(spin_limit: int = 1000, stream=None) -> int:
    """Run the bounded-wait self-test and return the status that
    ``device_status`` then reports (DEVSCAN_ERR_TIMEOUT = 4 expected)."""
    _lib.check(load().devscan_selftest_stalled_wait(int(spin_limit), _stream_handle(stream)),
               "devscan_selftest_stalled_wait")
    return device_status(stream)
