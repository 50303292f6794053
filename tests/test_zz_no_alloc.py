"""The allocation-free int32 exclusive scan, called through the C ABI.

scan_exclusive_i32_noalloc serves callers that cannot allocate device
memory: code whose GPU memory belongs to another allocator (a framework's
caching pool that has reserved the device) and code that must not allocate
once it is running.  Its scratch is one fixed array inside the library,
shared by every call.  These tests check, element by element:

* its results against the serial oracle (the exclusive scan of geek-doc.cn
  "并行前缀和 scan ..." section 一: z[0] is the identity, z[i] folds
  x[0 .. i-1]) and against the regular scan_exclusive_i32 entry point
  (integer scans are exact, so both must agree bit for bit);
* at the array's limit (2^28 elements: every tile status slot in use) and
  just below it, for add, max and xor;
* on calls in a row that share the array, a large one followed by a small
  one and another large one on different data (status words left by an
  earlier call must read as "not ready" through their epoch tag);
* on the scalar path (pointers 4-byte but not 16-byte aligned) and in place;
* that a call on a stream the library has never seen allocates no device
  memory.

This file is collected last so that a failure here cannot hide any other
test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

MAX_N = 1 << 28   # DEVSCAN_NOALLOC_MAX_N
OPS = {"add": 0, "max": 1, "xor": 2}


@pytest.fixture(scope="module")
def lib():
    from stream_compaction_device_gb300 import _lib
    return _lib.load()


def _input(n: int, op: str, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    if op == "add":
        return rng.integers(0, 10, n, dtype=np.int32)
    return rng.integers(-2**31, 2**31, n, dtype=np.int32)


def _noalloc(lib, d_in: torch.Tensor, d_out: torch.Tensor, n: int, op: str, stream=None):
    s = (stream or torch.cuda.current_stream()).cuda_stream
    assert lib.scan_exclusive_i32_noalloc(d_in.data_ptr(), d_out.data_ptr(), n, OPS[op], s) == 0


def _regular(lib, d_in: torch.Tensor, n: int, op: str) -> torch.Tensor:
    ref = torch.empty(n, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.scan_exclusive_i32(d_in.data_ptr(), ref.data_ptr(), n, OPS[op], s) == 0
    return ref


def _assert_equal(got: np.ndarray, ref: np.ndarray, what: str):
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at {bad[0]}: got {got[bad[0]]} want {ref[bad[0]]}"


def test_noalloc_call_allocates_nothing(lib):
    """Called alone on streams the library has not seen, before the regular
    entry point in this test: the result equals the oracle's, and the
    device's free memory is the same before and after the second call (the
    first call on a device may load the library's module, whose static
    array is part of the library, and looks up that array's address)."""
    x = _input(1_000_003, "add", 7)
    want = oracle.scan(x, "add", False)
    d_in = torch.from_numpy(x).cuda()
    outs = [torch.full_like(d_in, -1) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    _noalloc(lib, d_in, outs[0], x.size, "add", streams[0])
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    reserved_before = torch.cuda.memory_reserved()
    _noalloc(lib, d_in, outs[1], x.size, "add", streams[1])
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, f"device free memory changed by {free_before - free_after} bytes"
    assert torch.cuda.memory_reserved() == reserved_before
    for out in outs:
        _assert_equal(out.cpu().numpy(), want, "first calls")


@pytest.mark.parametrize("op", ["add", "max", "xor"])
def test_noalloc_at_the_limit_large_small_large(lib, op):
    """2^28 on one input, 12,293, 2^28 on another input, then 2^28 - 5 on
    the first: each against the oracle and the regular entry point."""
    seeds = {"add": 10, "max": 20, "xor": 30}[op]
    x1 = _input(MAX_N, op, seeds)
    x2 = _input(MAX_N, op, seeds + 1)
    small = _input(12_293, op, seeds + 2)
    want1 = oracle.scan(x1, op, False)
    cases = [(x1, MAX_N, want1), (small, small.size, oracle.scan(small, op, False)),
             (x2, MAX_N, oracle.scan(x2, op, False)), (x1, MAX_N - 5, want1[:MAX_N - 5])]
    d_out = torch.empty(MAX_N, dtype=torch.int32, device="cuda")
    for host, n, want in cases:
        d_in = torch.from_numpy(host[:n]).cuda()
        d_out.fill_(-1)
        _noalloc(lib, d_in, d_out, n, op)
        got = d_out[:n].cpu().numpy()
        _assert_equal(got, want, f"{op} n={n} against the oracle")
        ref = _regular(lib, d_in, n, op).cpu().numpy()
        _assert_equal(got, ref, f"{op} n={n} against scan_exclusive_i32")
        assert int(d_out[n:n + 1].cpu().item() if n < MAX_N else -1) == -1, "wrote past n"
        del d_in
    assert lib.devscan_device_status(torch.cuda.current_stream().cuda_stream) == 0


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_noalloc_scalar_path(lib, offset):
    """In and out 4-byte but not 16-byte aligned (offsets of 1-3 elements)."""
    for n, op in ((12_293, "max"), (1_000_003, "add"), (MAX_N - 5, "xor")):
        x = _input(n, op, 100 + offset)
        d_in = torch.zeros(n + offset, dtype=torch.int32, device="cuda")
        d_in[offset:] = torch.from_numpy(x).cuda()
        d_out = torch.full((n + offset,), -1, dtype=torch.int32, device="cuda")
        _noalloc(lib, d_in[offset:], d_out[offset:], n, op)
        got = d_out[offset:].cpu().numpy()
        _assert_equal(got, oracle.scan(x, op, False), f"offset {offset} n={n}")
        _assert_equal(got, _regular(lib, d_in[offset:], n, op).cpu().numpy(), f"offset {offset} n={n} regular")
        assert torch.all(d_out[:offset] == -1), "wrote before out"
        del d_in, d_out


def test_noalloc_in_place(lib):
    """in == out, aligned and not."""
    for n, offset in ((1_000_003, 0), ((1 << 22) + 3, 0), (300_001, 1)):
        x = _input(n, "add", n)
        d = torch.zeros(n + offset, dtype=torch.int32, device="cuda")
        d[offset:] = torch.from_numpy(x).cuda()
        ref = _regular(lib, d[offset:], n, "add").cpu().numpy()
        _noalloc(lib, d[offset:], d[offset:], n, "add")
        got = d[offset:].cpu().numpy()
        _assert_equal(got, oracle.scan(x, "add", False), f"in place n={n} offset={offset}")
        _assert_equal(got, ref, f"in place n={n} offset={offset} regular")


def test_noalloc_rejects_oversized_input(lib):
    x = torch.zeros(16, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # the size check comes before any use of the pointers
    assert lib.scan_exclusive_i32_noalloc(x.data_ptr(), x.data_ptr(), MAX_N + 1, 0, stream) == 1
    assert lib.scan_exclusive_i32_noalloc(x.data_ptr(), x.data_ptr(), 0, 0, stream) == 0
    assert lib.scan_exclusive_i32_noalloc(x.data_ptr(), x.data_ptr(), 16, 7, stream) == 1
