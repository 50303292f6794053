"""Scan parity: the CUDA library (through its C ABI) against the CPU oracle,
element by element on the same seeded inputs.  Integer scans are bit-exact;
fp32 add is within |err_i| <= 1e-5 * sum_{j<=i} |x_j| of the fp64 oracle;
fp32 max is bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_f32_within, from_dev, to_dev

pytestmark = pytest.mark.gpu

TILE = 4096
SIZES = [1, 2, 3, 4, 5, 7, 31, 32, 33, 127, 128, 129, 511, 512, 513, 1023, 1024, 1025,
         TILE - 1, TILE, TILE + 1, 2 * TILE - 3, 3 * TILE + 5, 65_536, 65_537, 262_147, 1_000_003]
CASES = [(np.int32, "add"), (np.int32, "max"), (np.int32, "xor"),
         (np.uint32, "add"), (np.uint32, "max"), (np.uint32, "xor"),
         (np.float32, "add"), (np.float32, "max")]


@pytest.fixture(scope="module")
def ds():
    import stream_compaction_device_gb300 as m
    m.load()
    return m


def gpu_scan(ds, x: np.ndarray, op: str, inclusive: bool, inplace=False, offset=0):
    d = to_dev(np.concatenate([np.zeros(offset, x.dtype), x]) if offset else x)
    if offset:
        d = d[offset:]
    out = d if inplace else None
    fn = ds.scan_inclusive if inclusive else ds.scan_exclusive
    y = fn(d, out=out, op=op, as_uint32=(x.dtype == np.uint32))
    torch.cuda.synchronize()
    return from_dev(y, x.dtype)


def check(ds, x, op, inclusive, **kw):
    got = gpu_scan(ds, x, op, inclusive, **kw)
    ref = oracle.scan(x, op, inclusive)
    if x.dtype == np.float32 and op == "add":
        assert_f32_within(got, ref, oracle.abs_prefix(x), f"n={x.size}")
    elif x.dtype == np.float32:
        assert np.array_equal(got.astype(np.float64), ref), f"n={x.size}"
    else:
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, f"n={x.size} op={op} incl={inclusive}: first mismatch at {bad[0]}"


@pytest.mark.parametrize("dtype,op", CASES, ids=lambda v: getattr(v, "__name__", v))
@pytest.mark.parametrize("inclusive", [True, False], ids=["incl", "excl"])
def test_scan_sizes(ds, dtype, op, inclusive):
    from stream_compaction_device_gb300 import workloads as wl
    for n in SIZES:
        check(ds, wl.random_input(dtype, n, seed=n, op=op), op, inclusive)


def test_worked_example(ds, golden):
    g = golden("worked_example.txt")
    x = np.array(g["x"], dtype=np.int32)
    assert gpu_scan(ds, x, "add", True).tolist() == g["inclusive"]
    assert gpu_scan(ds, x, "add", False).tolist() == g["exclusive"]


def test_empty(ds):
    x = torch.empty(0, dtype=torch.int32, device="cuda")
    assert ds.scan_inclusive(x).numel() == 0
    assert ds.scan_exclusive(x, op="max").numel() == 0


@pytest.mark.parametrize("inclusive", [True, False])
def test_in_place(ds, inclusive):
    from stream_compaction_device_gb300 import workloads as wl
    for n in (5, TILE + 1, 300_001):
        check(ds, wl.random_input(np.int32, n, 7, "add"), "add", inclusive, inplace=True)
        check(ds, wl.random_input(np.float32, n, 8, "add"), "add", inclusive, inplace=True)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_pointers(ds, offset):
    """in/out 4-byte but not 16-byte aligned take the scalar path."""
    from stream_compaction_device_gb300 import workloads as wl
    for n in (1, 33, TILE + 7, 60_001, 100_003):
        check(ds, wl.random_input(np.int32, n, n, "add"), "add", False, offset=offset)
        check(ds, wl.random_input(np.uint32, n, n, "max"), "max", True, offset=offset)
        check(ds, wl.random_input(np.float32, n, n, "add"), "add", True, offset=offset)


def test_int32_wraps(ds):
    x = np.full(10_000, 2**30, dtype=np.int32)
    check(ds, x, "add", True)
    check(ds, x, "add", False)


@pytest.mark.parametrize("mode", ["lookback", "rts", "pipelined", "l2"])
def test_carry_modes(ds, mode):
    """Every inter-block carry path gives the oracle's results."""
    from stream_compaction_device_gb300 import workloads as wl
    ds.set_carry_mode(mode)
    try:
        for dtype, op in CASES:
            for n in (1, 5, TILE, 2 * TILE + 1, 8192 * 3 + 7, 16384 * 152 + 9, 1_000_003, (1 << 21) + 17):
                for inclusive in (True, False):
                    check(ds, wl.random_input(dtype, n, n + 1, op), op, inclusive)
    finally:
        ds.set_carry_mode("default")


def test_reduce_then_scan_at_full_size(ds):
    """The reduce-then-scan carry at 2^28 elements, the size the benchmark
    times it at (65,536 tile totals scanned by one block)."""
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.brackets()
    ds.set_carry_mode("rts")
    try:
        got = gpu_scan(ds, x, "add", False)
    finally:
        ds.set_carry_mode("default")
    assert np.array_equal(got, oracle.scan(x, "add", False))
    assert ds.device_status() == 0


def test_default_size_boundaries(ds):
    """Sizes around the default's switches between the cluster scan, the
    one-tile kernel, the L2-resident scan and the pipeline (2^16, 2^17 and
    2^24), ragged blocks and chunks included."""
    from stream_compaction_device_gb300 import workloads as wl
    for n in (8191, 8192, 8193, 7 * 8192 + 1, (1 << 16) - 1, 1 << 16, (1 << 16) + 1,
              (1 << 17) - 1, 1 << 17, (1 << 17) + 4097, 3 * (1 << 20) + 1, (1 << 24) - 3, 1 << 24, (1 << 24) + 1):
        check(ds, wl.random_input(np.int32, n, n, "add"), "add", False)
        check(ds, wl.random_input(np.float32, n, n + 1, "add"), "add", True)
        check(ds, wl.random_input(np.uint32, n, n + 2, "max"), "max", False)


@pytest.mark.parametrize("mode", ["default", "lookback", "l2"])
def test_repeated_runs_identical(ds, mode):
    """Integer results do not depend on block timing: 50 launches, one answer."""
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.random_input(np.int32, (1 << 22) + 3, 11, "add")
    d = to_dev(x)
    ref = torch.from_numpy(oracle.scan(x, "add", False)).cuda()
    out = torch.empty_like(d)
    ds.set_carry_mode(mode)
    try:
        for _ in range(50):
            ds.scan_exclusive(d, out)
            assert torch.equal(out, ref)
    finally:
        ds.set_carry_mode("default")
    assert ds.device_status() == 0


def test_workspace_growth_and_streams(ds):
    from stream_compaction_device_gb300 import workloads as wl
    for n in (100, 5_000_001, 100, 2_000_000):
        check(ds, wl.random_input(np.int32, n, n, "xor"), "xor", True)
    s = torch.cuda.Stream()
    x = wl.random_input(np.int32, 3_000_001, 5, "add")
    with torch.cuda.stream(s):
        d = to_dev(x)
        y = ds.scan_inclusive(d, stream=s)
    s.synchronize()
    assert np.array_equal(y.cpu().numpy(), oracle.scan(x, "add", True))
    ds.stream_release(s)
    assert ds.device_status(s) == 0


def test_bounded_wait_reports_timeout(ds):
    """A look-back whose predecessor never publishes gives up and reports
    DEVSCAN_ERR_TIMEOUT; the stream stays usable afterwards."""
    assert ds.device_status() == 0
    assert ds.selftest_stalled_wait(2000) == 4
    assert ds.device_status() == 0
    check(ds, np.arange(100_000, dtype=np.int32), "add", True)


# ---------------------------------------------------------------------------
# full-size workloads, in the configuration the benchmark times
# ---------------------------------------------------------------------------
def test_config_small_digits(ds):
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.small_digits()
    check(ds, x, "add", True)
    check(ds, x, "add", False)


def test_config_unit_floats(ds):
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.unit_floats()
    check(ds, x, "add", True)
    check(ds, x, "add", False)


def test_config_sweep_brackets(ds):
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.brackets()
    got_incl = gpu_scan(ds, x, "add", True)
    ref_incl = oracle.scan(x, "add", True)
    assert np.array_equal(got_incl, ref_incl)
    assert oracle.bracket_flags(got_incl) == oracle.bracket_flags(ref_incl)
    del got_incl, ref_incl
    assert np.array_equal(gpu_scan(ds, x, "add", False), oracle.scan(x, "add", False))


def test_config_sweep_max(ds):
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.max_values()
    assert np.array_equal(gpu_scan(ds, x, "max", True), oracle.scan(x, "max", True))


def test_config_sweep_xor(ds):
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.xor_values()
    assert np.array_equal(gpu_scan(ds, x, "xor", True), oracle.scan(x, "xor", True))


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_entry(ds, pinned):
    """scan_{inclusive,exclusive}_host_T: host array in, host array out, the
    copies and the scan queued by the library on one stream; in place on
    the host and on the device too."""
    from stream_compaction_device_gb300 import workloads as wl
    for dtype, op in CASES:
        for n in (1, 4097, 1_000_003):
            x = wl.random_input(dtype, n, n + 5, op)
            hx = torch.from_numpy(x.view(np.int32) if dtype == np.uint32 else x)
            if pinned:
                hx = hx.pin_memory()
            for inclusive in (True, False):
                got = ds.scan_host(hx, inclusive=inclusive, op=op, as_uint32=dtype == np.uint32).numpy()
                got = got.view(np.uint32) if dtype == np.uint32 else got
                ref = oracle.scan(x, op, inclusive)
                if dtype == np.float32 and op == "add":
                    assert_f32_within(got, ref, oracle.abs_prefix(x), f"host n={n}")
                elif dtype == np.float32:
                    assert np.array_equal(got.astype(np.float64), ref)
                else:
                    assert np.array_equal(got, ref), (dtype, op, n, inclusive)
    # in place: one host array, one device buffer
    x = wl.random_input(np.int32, 300_001, 3, "add")
    h = torch.from_numpy(x.copy())
    if pinned:
        h = h.pin_memory()
    d = torch.empty(x.size, dtype=torch.int32, device="cuda")
    ds.scan_host(h, inclusive=False, out_host=h, work=(d, d))
    assert np.array_equal(h.numpy(), oracle.scan(x, "add", False))
