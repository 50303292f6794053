"""Parity of the fused operations against the CPU oracle, bit-exact:
compaction with the predicate (x > t) evaluated on the device, and the
bracket check fused into the inclusive add-scan (the scanned array, the
negative-prefix answer and the final sum)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import from_dev, to_dev

pytestmark = pytest.mark.gpu

I32_MIN, I32_MAX = -2**31, 2**31 - 1
SIZES = [1, 2, 3, 5, 15, 16, 17, 127, 128, 129, 4095, 4096, 4097, 8191, 8192, 8193, 3 * 8192 + 5,
         65_537, 300_007, 524_288, 524_291]


@pytest.fixture(scope="module")
def ds():
    import stream_compaction_device_gb300 as m
    m.load()
    return m


@pytest.fixture(params=["default", "lookback", "pipelined", "l2"])
def mode(request, ds):
    ds.set_carry_mode(request.param)
    yield request.param
    ds.set_carry_mode("default")


# ---------------------------------------------------------------------------
# compaction, predicate in the kernel
# ---------------------------------------------------------------------------
def gpu_compact_gt(ds, v: np.ndarray, t: int, voff=0, ooff=0):
    dv = to_dev(np.concatenate([np.zeros(voff, np.int32), v]))[voff:]
    out = torch.full((v.size + ooff + 8,), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ds.compact_greater(dv, t, out=out[ooff:ooff + max(v.size, 1)], count=cnt)
    torch.cuda.synchronize()
    k = int(cnt.item())
    host = out.cpu().numpy()
    assert np.all(host[:ooff] == -7) and np.all(host[ooff + k:] == -7), "write outside the kept range"
    return host[ooff:ooff + k]


def check_compact_gt(ds, v, t, **kw):
    got = gpu_compact_gt(ds, v, t, **kw)
    ref = oracle.compact(v, (v > np.int32(t)).astype(np.uint8))
    assert got.size == ref.size, f"count {got.size} != {ref.size} (n={v.size}, t={t})"
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"n={v.size} t={t}: first mismatch at {bad[0]}"


@pytest.mark.parametrize("t", [I32_MIN, -2_104_533_976, -1, 0, 2_104_533_974, I32_MAX])
def test_compact_gt_sizes(ds, mode, t):
    rng = np.random.default_rng(31)
    for n in SIZES:
        v = rng.integers(I32_MIN, I32_MAX + 1, n, dtype=np.int32)
        v[: min(n, 4)] = np.array([t, t + 1 if t < I32_MAX else t, I32_MIN, I32_MAX], np.int64)[: min(n, 4)]
        check_compact_gt(ds, v, t)


@pytest.mark.parametrize("voff,ooff", [(1, 0), (0, 1), (2, 3), (3, 2)])
def test_compact_gt_unaligned(ds, mode, voff, ooff):
    rng = np.random.default_rng(voff * 10 + ooff)
    for n in (1, 77, 8192 + 3, 200_001, 600_001):
        v = rng.integers(I32_MIN, I32_MAX + 1, n, dtype=np.int32)
        check_compact_gt(ds, v, -1, voff=voff, ooff=ooff)


def test_compact_gt_empty(ds):
    v = torch.empty(0, dtype=torch.int32, device="cuda")
    cnt = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    ds.compact_greater(v, 0, out=torch.empty(1, dtype=torch.int32, device="cuda"), count=cnt)
    assert int(cnt.item()) == 0


def test_compact_gt_worked_example(ds, golden):
    g = golden("worked_example.txt")
    x = np.array(g["x"], dtype=np.int32)
    assert gpu_compact_gt(ds, x, g["predicate_threshold"][0]).tolist() == g["compacted"]


@pytest.mark.parametrize("sel", [0.01, 0.50, 0.99])
def test_config_compact_gt(ds, sel):
    from stream_compaction_device_gb300 import workloads as wl
    v = wl.compaction_values()
    check_compact_gt(ds, v, wl.threshold_for(sel))
    assert ds.device_status() == 0


def drain_capture_backoff(ds, n=1 << 24):
    """After a capture gives up, the stream's next 16 calls skip it and run
    the pipeline; 17 calls that keep nothing bring the stream back to
    capturing (the 17th captures)."""
    v = torch.full((n,), -5, dtype=torch.int32, device="cuda")
    out = torch.empty_like(v)
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    for _ in range(17):
        ds.compact_greater(v, 0, out=out, count=cnt)
    assert int(cnt.item()) == 0


@pytest.mark.parametrize("sel", [0.0, 0.001, 0.05, 0.09, 0.095, 0.10, 0.105, 0.11, 0.13, 0.20, 1.0])
def test_compact_gt_capture_band(ds, sel):
    """The default form on the 2^26 workload around the selectivity where the
    one-pass capture stops fitting in shared memory (about 10% kept): each
    call either captures and writes, or gives up and the kernel goes on as
    the pipeline (and the next calls skip the capture); the
    result is the oracle's either way."""
    from stream_compaction_device_gb300 import workloads as wl
    v = wl.compaction_values()
    t = {0.0: I32_MAX, 1.0: I32_MIN}.get(sel)
    drain_capture_backoff(ds)
    for _ in range(2):   # and again, after whichever outcome the first call had
        check_compact_gt(ds, v, wl.threshold_for(sel) if t is None else t)
    assert ds.device_status() == 0


@pytest.mark.parametrize("pattern", ["dense_tail", "dense_late_in_ranges", "dense_head", "alternating"])
def test_compact_gt_capture_gives_up(ds, pattern):
    """Inputs whose kept values bunch up where a one-pass capture meets them
    late or early: the capture gives up part-way and the kernel goes on as
    the pipeline; a sparse call during the back-off that
    follows, and one after it, get the oracle's result too."""
    n = 1 << 24
    rng = np.random.default_rng(sum(map(ord, pattern)))
    v = rng.integers(-1000, 0, n, dtype=np.int32)                 # nothing kept at threshold 0 ...
    i = np.arange(n)
    if pattern == "dense_tail":                                    # ... except the last 3% (all kept)
        dense = i >= n - n // 32
    elif pattern == "dense_late_in_ranges":                        # the last fifth of every 16,384
        dense = (i % 16384) >= 13107
    elif pattern == "dense_head":                                  # the first 3%
        dense = i < n // 32
    else:                                                          # every other 4,096 (half kept)
        dense = ((i // 4096) % 2) == 1
    v[dense] = rng.integers(1, 1000, int(dense.sum()), dtype=np.int32)
    sparse = rng.random(n) < 0.01
    v[sparse] = rng.integers(1, 1000, int(sparse.sum()), dtype=np.int32)
    drain_capture_backoff(ds)
    check_compact_gt(ds, v, 0)
    w = rng.integers(-1000, 1000, n, dtype=np.int32)
    check_compact_gt(ds, w, 979)                                   # about 1% kept, during the back-off
    drain_capture_backoff(ds)
    check_compact_gt(ds, w, 979)                                   # and captured again
    assert ds.device_status() == 0


@pytest.mark.parametrize("sel", [0.0, 0.01, 0.50, 0.99, 1.0])
def test_config_compact_gt_two_launch(ds, sel):
    """The two-launch form (a count of every 512-element part from the
    values, then a warp per part) on the 2^26 workload, and with nothing or
    everything kept."""
    from stream_compaction_device_gb300 import workloads as wl
    v = wl.compaction_values()
    t = {0.0: I32_MAX, 1.0: I32_MIN}.get(sel)
    ds.set_carry_mode("l2")
    try:
        check_compact_gt(ds, v, wl.threshold_for(sel) if t is None else t)
    finally:
        ds.set_carry_mode("default")
    assert ds.device_status() == 0


# ---------------------------------------------------------------------------
# bracket check fused into the scan
# ---------------------------------------------------------------------------
def gpu_bracket(ds, x: np.ndarray, store=True, xoff=0, ooff=0, in_place=False):
    dx = to_dev(np.concatenate([np.zeros(xoff, np.int32), x]))[xoff:]
    res = torch.full((2,), -5, dtype=torch.int32, device="cuda")
    out = None
    if in_place:
        out = dx
    elif store:
        out = torch.full((x.size + ooff,), -9, dtype=torch.int32, device="cuda")[ooff:]
    got_out, _ = ds.bracket_scan(dx, out=out, result=res, store=store or in_place)
    torch.cuda.synchronize()
    r = res.cpu().numpy()
    incl = got_out.cpu().numpy() if got_out is not None else None
    return incl, bool(r[0]), int(r[1])


def check_bracket(ds, x, **kw):
    ref = oracle.scan(x, "add", True)
    neg, _ = oracle.bracket_flags(ref)
    final = int(ref[-1]) if x.size else 0
    incl, got_neg, got_final = gpu_bracket(ds, x, **kw)
    assert (got_neg, got_final) == (neg, final), f"n={x.size}: ({got_neg}, {got_final}) != ({neg}, {final})"
    if incl is not None:
        bad = np.nonzero(incl != ref)[0]
        assert bad.size == 0, f"n={x.size}: scan differs first at {bad[0]}"


def dyck(m: int, rng) -> np.ndarray:
    """A random balanced sequence of m pairs: shuffle, then rotate to the
    first minimum of the running sum (the cycle lemma makes the rotation
    nonnegative throughout)."""
    x = np.array([1] * m + [-1] * m, dtype=np.int32)
    rng.shuffle(x)
    c = np.cumsum(x)
    k = int(np.argmin(c)) + 1 if x.size else 0
    return np.roll(x, -k)


@pytest.mark.parametrize("store", [True, False])
def test_bracket_sizes(ds, mode, store):
    rng = np.random.default_rng(41)
    for n in SIZES:
        x = (2 * rng.integers(0, 2, n) - 1).astype(np.int32)
        check_bracket(ds, x, store=store)


@pytest.mark.parametrize("store", [True, False])
def test_bracket_cases(ds, mode, store):
    rng = np.random.default_rng(42)
    for m in (1, 2, 2048, 4096, 150_000, 300_000):
        x = dyck(m, rng)
        assert np.all(np.cumsum(x) >= 0) and x.sum() == 0
        check_bracket(ds, x, store=store)                     # balanced
        y = x.copy()
        y[-2:] = y[-2:][::-1]                                  # last two swapped
        check_bracket(ds, y, store=store)
        z = np.concatenate([x[1:], x[:1]])                     # starts with ')' : negative prefix at once
        check_bracket(ds, z, store=store)
        w = x.copy()
        w[-1] = 1                                              # final sum 2, never negative
        check_bracket(ds, w, store=store)
        u = x.copy()
        u[x.size // 2:] = -u[x.size // 2:]                     # a deep negative dip in the middle
        check_bracket(ds, u, store=store)


def test_bracket_wrap_and_weights(ds, mode):
    rng = np.random.default_rng(43)
    for n in (1, 4097, 70_001, 600_001):
        x = rng.integers(I32_MIN, I32_MAX + 1, n, dtype=np.int32)   # prefixes wrap modulo 2^32
        check_bracket(ds, x)
        check_bracket(ds, x, store=False)
    x = np.full(600_001, I32_MAX // 4, dtype=np.int32)             # wraps to negative after 5 terms
    check_bracket(ds, x)


@pytest.mark.parametrize("xoff,ooff", [(1, 0), (0, 1), (3, 2)])
def test_bracket_unaligned(ds, mode, xoff, ooff):
    rng = np.random.default_rng(xoff + 5 * ooff)
    for n in (1, 99, 4096 + 5, 600_003):
        x = (2 * rng.integers(0, 2, n) - 1).astype(np.int32)
        check_bracket(ds, x, xoff=xoff, ooff=ooff)
        check_bracket(ds, x, store=False, xoff=xoff)


@pytest.mark.parametrize("carry", ["default", "l2"])
def test_bracket_check_only(ds, carry):
    """The check without the scanned array: in the default mode from 2^17
    elements (and in mode "l2" at every size) one cooperative launch folds
    (sum, lowest prefix, highest prefix) runs; chunks whose prefixes cross a
    wrap of int32 are checked again element by element."""
    ds.set_carry_mode(carry)
    try:
        rng = np.random.default_rng(46)
        sizes = [(1 << 17) - 1, 1 << 17, (1 << 17) + 3, 300_007, 16_384 * 152 + 5, 1_000_003, (1 << 22) + 1]
        if carry == "l2":
            sizes = [1, 5, 513, 4097, 16_385] + sizes[:3]
        for n in sizes:
            x = (2 * rng.integers(0, 2, n) - 1).astype(np.int32)
            check_bracket(ds, x, store=False)                      # random walk: dips below zero
            m = n // 2
            d = dyck(m, rng)
            if n % 2:
                d = np.concatenate([d, np.array([1], np.int32)])
            check_bracket(ds, d, store=False)                      # never negative
            z = np.concatenate([d[1:], d[:1]])
            check_bracket(ds, z, store=False)
            big = rng.integers(I32_MIN, I32_MAX + 1, n, dtype=np.int32)
            check_bracket(ds, big, store=False)                    # prefixes wrap many times
            up = np.full(n, 1 << 20, dtype=np.int32)
            check_bracket(ds, up, store=False)                     # exact prefix passes 2^31: wraps negative
            down = np.full(n, -(1 << 20), dtype=np.int32)
            down[0] = 5
            check_bracket(ds, down, store=False)
        assert ds.device_status() == 0
    finally:
        ds.set_carry_mode("default")


def test_bracket_in_place(ds, mode):
    rng = np.random.default_rng(44)
    for n in (5, 8193, 600_001):
        x = (2 * rng.integers(0, 2, n) - 1).astype(np.int32)
        check_bracket(ds, x, in_place=True)


def test_bracket_empty(ds):
    x = torch.empty(0, dtype=torch.int32, device="cuda")
    res = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    ds.bracket_scan(x, result=res, store=False)
    assert res.cpu().tolist() == [0, 0]


def test_config_bracket(ds):
    """The 2^28-element +1/-1 sweep array: the check alone (read-only) and
    the scan with the check, against the oracle."""
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.brackets()
    ref = oracle.scan(x, "add", True)
    neg, _ = oracle.bracket_flags(ref)
    want = (neg, int(ref[-1]))
    incl, got_neg, got_final = gpu_bracket(ds, x, store=False)
    assert (got_neg, got_final) == want
    incl, got_neg, got_final = gpu_bracket(ds, x, store=True)
    assert (got_neg, got_final) == want
    assert np.array_equal(incl, ref)
    del incl, ref
    # a balanced array of the same size: neither answer may fire
    # "()" pairs, a random half of the 4-blocks nested as "(())"
    rng = np.random.default_rng(45)
    b = np.tile(np.array([1, -1], dtype=np.int32), x.size // 2)
    blocks = b.reshape(-1, 4)
    blocks[rng.random(blocks.shape[0]) < 0.5] = np.array([1, 1, -1, -1], dtype=np.int32)
    _, got_neg, got_final = gpu_bracket(ds, b, store=False)
    assert (got_neg, got_final) == (False, 0)
    assert ds.device_status() == 0
