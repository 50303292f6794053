"""Serial CPU oracle for the device-wide prefix scan and its two consumers.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
CUDA library never calls it, and it shares no code with the CUDA library:
the arithmetic lives in ``oracle.c`` (plain serial C loops, one per
definition on the pages), built with gcc into ``liboracle.so`` and called
through ctypes on NumPy arrays.

Pages followed (cited per routine in ``oracle.c``):

* geek-doc.cn "并行前缀和 scan: Hillis-Steele、Blelloch 与 warp shuffle 三种写法",
  section 一 -- inclusive/exclusive scan, compaction, radix split, brackets;
* lpnh.cn/news/2866224 "并行扫描 Scan/Prefix Sum", sections 2.1, 2.2, 3.3, 4.1,
  7.2 (segmented scan);
* pgsm.cn/news/414823 "SIMT数据依赖与并行前缀和", sections 4.1-4.2.

Every function here is pinned by ``tests/test_oracle_pins.py`` against the
pages' printed worked examples, brute force on tiny inputs, closed forms and
independent restatements.  The fp32 add scan is accumulated in fp64: its
parallel rounding pattern is bounded (tolerance), not pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_MT_SRC = os.path.join(_HERE, "mt_baseline.c")   # the multithreaded CPU baseline (not the oracle)
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

OPS = {"add": 0, "max": 1, "xor": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (no -ffast-math)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_MT_SRC)))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared", "-pthread", "-Wall",
               "-Wextra", "-o", tmp, _SRC, _MT_SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        for name in ("oracle_scan_i32", "oracle_scan_u32", "oracle_scan_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, sz, i, i]
            fn.restype = i
        for name in ("oracle_segscan_i32", "oracle_segscan_u32", "oracle_segscan_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp, sz, i, i]
            fn.restype = i
        lib.oracle_abs_prefix_f32.argtypes = [vp, vp, sz]
        lib.oracle_abs_prefix_f32.restype = None
        lib.oracle_seg_abs_prefix_f32.argtypes = [vp, vp, vp, sz]
        lib.oracle_seg_abs_prefix_f32.restype = None
        lib.oracle_compact_i32.argtypes = [vp, vp, vp, sz]
        lib.oracle_compact_i32.restype = ctypes.c_int64
        lib.oracle_split_bit_u32.argtypes = [vp, vp, i, sz]
        lib.oracle_split_bit_u32.restype = ctypes.c_int64
        lib.oracle_sort_lsd_u32.argtypes = [vp, vp, sz]
        lib.oracle_sort_lsd_u32.restype = None
        lib.oracle_bracket_flags.argtypes = [vp, sz, ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.oracle_bracket_flags.restype = None
        lib.mt_scan_excl_add_i32.argtypes = [vp, vp, sz, i]
        lib.mt_scan_excl_add_i32.restype = i
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _contig(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype).name}, got {a.dtype}")
    return np.ascontiguousarray(a)


def scan(x, op: str = "add", inclusive: bool = True) -> np.ndarray:
    """Serial inclusive or exclusive scan of ``x`` under ``op``.

    int32 and uint32 inputs give outputs of the same type (add wraps modulo
    2^32).  fp32 inputs give an fp64 reference: add is accumulated in fp64,
    max is exact.  Raises ``ValueError`` for an operator the type lacks
    (xor on fp32)."""
    x = np.asarray(x)
    code = OPS[op]
    lib = _load()
    if x.dtype == np.int32:
        x = np.ascontiguousarray(x)
        y = np.empty_like(x)
        rc = lib.oracle_scan_i32(_ptr(x), _ptr(y), x.size, code, int(inclusive))
    elif x.dtype == np.uint32:
        x = np.ascontiguousarray(x)
        y = np.empty_like(x)
        rc = lib.oracle_scan_u32(_ptr(x), _ptr(y), x.size, code, int(inclusive))
    elif x.dtype == np.float32:
        x = np.ascontiguousarray(x)
        y = np.empty(x.shape, dtype=np.float64)
        rc = lib.oracle_scan_f32(_ptr(x), _ptr(y), x.size, code, int(inclusive))
    else:
        raise TypeError(f"unsupported dtype {x.dtype}")
    if rc != 0:
        raise ValueError(f"operator {op!r} is not defined for {x.dtype}")
    return y


def segscan(x, heads, op: str = "add", inclusive: bool = True) -> np.ndarray:
    """Serial segmented scan: a nonzero ``heads[i]`` starts a new segment at
    i (element 0 always starts one) and the accumulator restarts from the
    operator's identity there.  Types and precision as :func:`scan`."""
    x = np.ascontiguousarray(np.asarray(x))
    heads = np.ascontiguousarray(np.asarray(heads, dtype=np.uint8))
    if heads.size != x.size:
        raise ValueError("x and heads differ in length")
    code = OPS[op]
    lib = _load()
    if x.dtype == np.int32:
        y = np.empty_like(x)
        rc = lib.oracle_segscan_i32(_ptr(x), _ptr(heads), _ptr(y), x.size, code, int(inclusive))
    elif x.dtype == np.uint32:
        y = np.empty_like(x)
        rc = lib.oracle_segscan_u32(_ptr(x), _ptr(heads), _ptr(y), x.size, code, int(inclusive))
    elif x.dtype == np.float32:
        y = np.empty(x.shape, dtype=np.float64)
        rc = lib.oracle_segscan_f32(_ptr(x), _ptr(heads), _ptr(y), x.size, code, int(inclusive))
    else:
        raise TypeError(f"unsupported dtype {x.dtype}")
    if rc != 0:
        raise ValueError(f"operator {op!r} is not defined for {x.dtype}")
    return y


def seg_abs_prefix(x, heads) -> np.ndarray:
    """fp64 running sum of |x_j| over the segment of i, j <= i: the fp32
    tolerance scale of the segmented scan."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    heads = np.ascontiguousarray(heads, dtype=np.uint8)
    s = np.empty(x.shape, dtype=np.float64)
    _load().oracle_seg_abs_prefix_f32(_ptr(x), _ptr(heads), _ptr(s), x.size)
    return s


def abs_prefix(x) -> np.ndarray:
    """fp64 running sum of |x_j| for j <= i: the fp32 tolerance scale."""
    x = _contig(x, np.float32)
    s = np.empty(x.shape, dtype=np.float64)
    _load().oracle_abs_prefix_f32(_ptr(x), _ptr(s), x.size)
    return s


def compact(values, flags) -> np.ndarray:
    """Order-preserving compaction: the values whose flag is nonzero."""
    values = _contig(values, np.int32)
    flags = _contig(flags, np.uint8)
    if values.size != flags.size:
        raise ValueError("values and flags differ in length")
    out = np.empty_like(values)
    k = _load().oracle_compact_i32(_ptr(values), _ptr(flags), _ptr(out), values.size)
    return out[:k].copy()


def split_bit(keys, bit: int) -> tuple[np.ndarray, int]:
    """Stable partition of ``keys`` by bit ``bit``: zeros first.  Returns the
    partitioned keys and the number of zeros."""
    keys = _contig(keys, np.uint32)
    if not 0 <= bit <= 31:
        raise ValueError("bit must be in [0, 31]")
    out = np.empty_like(keys)
    zeros = _load().oracle_split_bit_u32(_ptr(keys), _ptr(out), bit, keys.size)
    return out, int(zeros)


def sort_lsd(keys) -> np.ndarray:
    """32-pass least-significant-bit-first radix sort by one-bit splits."""
    keys = _contig(keys, np.uint32).copy()
    tmp = np.empty_like(keys)
    _load().oracle_sort_lsd_u32(_ptr(keys), _ptr(tmp), keys.size)
    return keys


def bracket_flags(incl) -> tuple[bool, bool]:
    """(negative prefix seen, final sum nonzero) from an inclusive add-scan
    of a +1/-1 bracket sequence."""
    incl = _contig(incl, np.int32)
    neg, unb = ctypes.c_int(0), ctypes.c_int(0)
    _load().oracle_bracket_flags(_ptr(incl), incl.size, ctypes.byref(neg), ctypes.byref(unb))
    return bool(neg.value), bool(unb.value)


def identity(op: str, dtype) -> float | int:
    """The operator's identity: the first element of an exclusive scan."""
    dtype = np.dtype(dtype)
    if op in ("add", "xor"):
        return 0
    if dtype == np.int32:
        return int(np.iinfo(np.int32).min)
    if dtype == np.uint32:
        return 0
    return float("-inf")


def mt_scan_exclusive_add(x, threads: int | None = None) -> tuple[np.ndarray, int]:
    """The multithreaded CPU baseline (``mt_baseline.c``, not the oracle):
    blocked three-phase int32 exclusive add-scan on up to ``threads`` host
    threads (default: every core).  Returns (scan, threads used)."""
    x = _contig(x, np.int32)
    y = np.empty_like(x)
    t = threads if threads is not None else (os.cpu_count() or 1)
    used = _load().mt_scan_excl_add_i32(_ptr(x), _ptr(y), x.size, int(t))
    return y, int(used)
