"""ctypes binding of ``libdevscan.so`` (the C ABI in ``include/devscan.h``).

Argument marshalling only: every step of a scan, compaction or split runs in
the library's CUDA kernels.  There is no fallback: if the shared library is
missing, loading it raises ``DevscanError`` naming the build command.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdevscan.so")

OPS = {"add": 0, "max": 1, "xor": 2}
STATUS = {0: "DEVSCAN_OK", 1: "DEVSCAN_ERR_INVALID", 2: "DEVSCAN_ERR_UNSUPPORTED",
          3: "DEVSCAN_ERR_CUDA", 4: "DEVSCAN_ERR_TIMEOUT", 5: "DEVSCAN_ERR_NOMEM"}
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_NOMEM = range(6)

SCAN_SYMBOLS = [f"scan_{d}_{t}" for d in ("inclusive", "exclusive") for t in ("i32", "u32", "f32")]
HOST_SCAN_SYMBOLS = tuple(f"scan_{d}_host_{t}" for d in ("inclusive", "exclusive") for t in ("i32", "u32", "f32"))
CARRY_SCAN_SYMBOLS = tuple(f"scan_{d}_carry_{t}" for d in ("inclusive", "exclusive") for t in ("i32", "u32", "f32"))
REDUCE_SYMBOLS = ("reduce_i32", "reduce_u32", "reduce_f32")
SEGSCAN_SYMBOLS = tuple(f"segmented_scan_{d}_{t}" for d in ("inclusive", "exclusive")
                        for t in ("i32", "u32", "f32"))


class DevscanError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libdevscan.so once and declare every entry point's signature."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise DevscanError(ERR_CUDA, f"{LIB_PATH} is not built (run: python -m "
                                         "stream_compaction_device_gb300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, sz, i, u = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint
        for name in SCAN_SYMBOLS:
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, sz, i, vp]
            fn.restype = i
        for name in HOST_SCAN_SYMBOLS:
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, sz, i, vp, vp, vp]
            fn.restype = i
        for name in CARRY_SCAN_SYMBOLS:
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, sz, i, vp, vp]
            fn.restype = i
        for name in REDUCE_SYMBOLS:
            fn = getattr(lib, name)
            fn.argtypes = [vp, sz, i, vp, vp]
            fn.restype = i
        for name in SEGSCAN_SYMBOLS:
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp, sz, i, vp]
            fn.restype = i
        lib.compact_i32.argtypes = [vp, vp, vp, vp, sz, vp]
        lib.compact_i32.restype = i
        lib.split_bit_u32.argtypes = [vp, vp, i, sz, vp]
        lib.split_bit_u32.restype = i
        lib.radix_sort_u32.argtypes = [vp, vp, sz, vp]
        lib.radix_sort_u32.restype = i
        lib.compact_gt_i32.argtypes = [vp, ctypes.c_int32, vp, vp, sz, vp]
        lib.compact_gt_i32.restype = i
        lib.bracket_scan_i32.argtypes = [vp, vp, vp, sz, vp]
        lib.bracket_scan_i32.restype = i
        lib.radix_sort_digits_u32.argtypes = [vp, vp, sz, vp]
        lib.radix_sort_digits_u32.restype = i
        lib.devscan_device_status.argtypes = [vp]
        lib.devscan_device_status.restype = i
        lib.devscan_status_string.argtypes = [i]
        lib.devscan_status_string.restype = ctypes.c_char_p
        lib.devscan_stream_release.argtypes = [vp]
        lib.devscan_stream_release.restype = i
        lib.devscan_measure_set_carry_mode.argtypes = [i]
        lib.devscan_measure_set_carry_mode.restype = i
        lib.devscan_selftest_stalled_wait.argtypes = [u, vp]
        lib.devscan_selftest_stalled_wait.restype = i
        lib.scan_exclusive_i32_noalloc.argtypes = [vp, vp, sz, i, vp]
        lib.scan_exclusive_i32_noalloc.restype = i
        _lib = lib
        return lib


def check(status: int, what: str) -> None:
    if status != OK:
        raise DevscanError(status, what)
