"""The allocation-free int32 exclusive scan, called through the C ABI.

scan_exclusive_i32_noalloc serves callers that cannot allocate device
memory (their GPU memory belongs to another allocator, or they must not
allocate after start-up): its scratch is a fixed array inside the library.
Its results must equal those of the regular scan_exclusive_i32 entry point
bit for bit (integer scans are exact), on two calls in a row that share the
same scratch array.  This file is collected last so that a failure here
cannot hide any other test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

MAX_N = 1 << 28   # DEVSCAN_NOALLOC_MAX_N


@pytest.fixture(scope="module")
def lib():
    from stream_compaction_device_gb300 import _lib
    lib = _lib.load()
    fn = lib.scan_exclusive_i32_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return lib


def _both(lib, x: torch.Tensor, op: int):
    stream = torch.cuda.current_stream().cuda_stream
    ref = torch.empty_like(x)
    got = torch.full_like(x, -1)
    assert lib.scan_exclusive_i32(x.data_ptr(), ref.data_ptr(), x.numel(), op, stream) == 0
    assert lib.scan_exclusive_i32_noalloc(x.data_ptr(), got.data_ptr(), x.numel(), op, stream) == 0
    torch.cuda.synchronize()
    return ref, got


@pytest.mark.parametrize("op", [0, 1, 2], ids=["add", "max", "xor"])
def test_noalloc_matches_regular_entry_point_twice(lib, op):
    rng = np.random.default_rng(40 + op)
    for n in (3 * 4096 + 5, 1_000_003):       # two calls in a row on the shared scratch
        if op == 0:
            host = rng.integers(0, 10, n, dtype=np.int32)
        else:
            host = rng.integers(-2**31, 2**31, n, dtype=np.int32)
        x = torch.from_numpy(host).cuda()
        ref, got = _both(lib, x, op)
        assert torch.equal(ref, got), f"n={n} op={op}"


def test_noalloc_rejects_oversized_input(lib):
    x = torch.zeros(16, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # the size check comes before any use of the pointers
    assert lib.scan_exclusive_i32_noalloc(x.data_ptr(), x.data_ptr(), MAX_N + 1, 0, stream) == 1
    assert lib.scan_exclusive_i32_noalloc(x.data_ptr(), x.data_ptr(), 0, 0, stream) == 0
