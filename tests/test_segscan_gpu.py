"""Segmented scan parity: the CUDA library against the CPU oracle, bit-exact
for the integer types, within 1e-5 of each segment's |x| prefix for fp32
add; head patterns chosen to reach every carry path (no heads, a head
everywhere, heads on tile and tile-group boundaries, one head far from any
other)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import F32_RTOL, assert_f32_within, from_dev, to_dev

pytestmark = pytest.mark.gpu

CASES = [(np.int32, "add"), (np.int32, "max"), (np.int32, "xor"), (np.uint32, "add"), (np.uint32, "max"),
         (np.uint32, "xor"), (np.float32, "add"), (np.float32, "max")]
SIZES = [1, 2, 3, 5, 31, 32, 33, 127, 128, 129, 4095, 4096, 4097, 8191, 8192, 8193, 3 * 8192 + 5, 65_537,
         300_007, 524_288, 524_291]
PIPE_TILE = 8192
GROUP = 32 * PIPE_TILE   # tiles per look-back group word


@pytest.fixture(scope="module")
def ds():
    import stream_compaction_device_gb300 as m
    m.load()
    return m


@pytest.fixture(params=["lookback", "pipelined"])
def mode(request, ds):
    ds.set_carry_mode(request.param)
    yield request.param
    ds.set_carry_mode("default")


def values_for(dtype, op, n, rng):
    if dtype == np.float32:
        if op == "max":
            return (rng.standard_normal(n) * 1000).astype(np.float32)
        return rng.random(n, dtype=np.float32)
    if op == "add":
        return rng.integers(0, 10, n).astype(dtype)
    if dtype == np.int32:
        return rng.integers(-2**31, 2**31, n, dtype=np.int64).astype(np.int32)
    return rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)


def gpu_segscan(ds, x, heads, op, inclusive, xoff=0, hoff=0, ooff=0, in_place=False):
    dx = to_dev(np.concatenate([np.zeros(xoff, x.dtype), x]))[xoff:]
    dh = torch.from_numpy(np.concatenate([np.zeros(hoff, np.uint8), heads])).cuda()[hoff:]
    if in_place:
        out = dx
    else:
        out = torch.empty(x.size + ooff, dtype=dx.dtype, device="cuda")[ooff:]
    fn = ds.segmented_scan_inclusive if inclusive else ds.segmented_scan_exclusive
    fn(dx, dh, out=out, op=op, as_uint32=(x.dtype == np.uint32))
    torch.cuda.synchronize()
    return from_dev(out, x.dtype)


def check(ds, x, heads, op, inclusive, **kw):
    got = gpu_segscan(ds, x, heads, op, inclusive, **kw)
    ref = oracle.segscan(x, heads, op, inclusive)
    what = f"n={x.size} {x.dtype} {op} {'incl' if inclusive else 'excl'}"
    if x.dtype == np.float32 and op == "add":
        assert_f32_within(got, ref, oracle.seg_abs_prefix(x, heads), what)
    else:
        bad = np.nonzero(got.astype(ref.dtype) != ref)[0]
        assert bad.size == 0, f"{what}: first mismatch at {bad[0]}: got {got[bad[0]]} ref {ref[bad[0]]}"


@pytest.mark.parametrize("dtype,op", CASES, ids=lambda c: str(c))
@pytest.mark.parametrize("inclusive", [True, False])
def test_segscan_sizes(ds, mode, dtype, op, inclusive):
    rng = np.random.default_rng(51)
    for n in SIZES:
        x = values_for(dtype, op, n, rng)
        h = (rng.random(n) < 0.002).astype(np.uint8)
        check(ds, x, h, op, inclusive)


@pytest.mark.parametrize("inclusive", [True, False])
def test_segscan_head_patterns(ds, mode, inclusive):
    rng = np.random.default_rng(52)
    n = 3 * GROUP + 12_345
    x = rng.integers(0, 10, n).astype(np.int32)
    patterns = {
        "none": np.zeros(n, np.uint8),
        "all": np.ones(n, np.uint8),
        "dense": (rng.random(n) < 0.5).astype(np.uint8),
        "sparse": (rng.random(n) < 1e-5).astype(np.uint8),
        "no head at 0": np.concatenate([[0], (rng.random(n - 1) < 1e-3)]).astype(np.uint8),
        "last element only": np.eye(1, n, n - 1, dtype=np.uint8)[0],
        "middle only": np.eye(1, n, n // 2 + 7, dtype=np.uint8)[0],
        "values 2..255": ((rng.random(n) < 0.01) * rng.integers(2, 256, n)).astype(np.uint8),
    }
    # heads at the first / last element of one-tile and pipeline tiles, and
    # inside the tile that closes a group of 32 (its group word carries it)
    edges = np.zeros(n, np.uint8)
    for t in (1, 5, 31, 32, 63, 64, 95):
        for off in (0, PIPE_TILE - 1, 100):
            if t * PIPE_TILE + off < n:
                edges[t * PIPE_TILE + off] = 1
    for t in (3, 9, 190):
        edges[t * 4096] = 1
        edges[t * 4096 + 4095] = 1
    patterns["tile and group edges"] = edges
    closing = np.zeros(n, np.uint8)
    closing[31 * PIPE_TILE + 4000] = 1   # only inside the first group's closing tile
    closing[2 * GROUP + 31 * PIPE_TILE + 8000] = 1
    patterns["group-closing tiles only"] = closing
    # the pipelined policy splits a tile into 512-element parts: heads at a
    # part's first and last element, in alternate parts only, and in the
    # tile's last part only
    parts = np.zeros(n, np.uint8)
    for t in (0, 2, 7, 40):
        for q in (0, 1, 7, 15):
            for off in (0, 511):
                e = t * PIPE_TILE + q * 512 + off
                if e < n:
                    parts[e] = 1
    patterns["part edges"] = parts
    alt = np.zeros(n, np.uint8)
    alt[(np.arange(n) // 512) % 2 == 1] = (rng.random(n) < 0.01)[(np.arange(n) // 512) % 2 == 1]
    patterns["alternate parts"] = alt
    last_part = np.zeros(n, np.uint8)
    for t in range(0, n // PIPE_TILE, 3):
        last_part[t * PIPE_TILE + 15 * 512 + 100] = 1
    patterns["last part of every third tile"] = last_part
    for name, h in patterns.items():
        got = gpu_segscan(ds, x, h, "add", inclusive)
        ref = oracle.segscan(x, h, "add", inclusive)
        assert ds.device_status() == 0, f"{name}: a bounded wait ran out"
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, f"{name}: first mismatch at {bad[0]}"


@pytest.mark.parametrize("xoff,hoff,ooff", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1), (0, 4, 0)])
def test_segscan_unaligned(ds, mode, xoff, hoff, ooff):
    rng = np.random.default_rng(xoff * 100 + hoff * 10 + ooff)
    for n in (1, 77, 4096 + 3, 600_001):
        x = rng.integers(0, 10, n).astype(np.int32)
        h = (rng.random(n) < 0.01).astype(np.uint8)
        for inclusive in (True, False):
            check(ds, x, h, "add", inclusive, xoff=xoff, hoff=hoff, ooff=ooff)


def test_segscan_in_place(ds, mode):
    rng = np.random.default_rng(53)
    for n in (9, 8193, 600_001):
        x = rng.integers(-2**31, 2**31, n, dtype=np.int64).astype(np.int32)
        h = (rng.random(n) < 0.01).astype(np.uint8)
        check(ds, x, h, "max", True, in_place=True)
        check(ds, x, h, "add", False, in_place=True)


def test_segscan_empty_and_errors(ds):
    x = torch.empty(0, dtype=torch.int32, device="cuda")
    h = torch.empty(0, dtype=torch.uint8, device="cuda")
    assert ds.segmented_scan_inclusive(x, h).numel() == 0
    xf = torch.zeros(8, dtype=torch.float32, device="cuda")
    hf = torch.zeros(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(Exception):
        ds.segmented_scan_inclusive(xf, hf, op="xor")


def test_segscan_worked_example(ds, golden):
    g = golden("segmented.txt")
    x = np.array(g["x"], dtype=np.int32)
    h = np.array(g["heads"], dtype=np.uint8)
    assert gpu_segscan(ds, x, h, "add", True).tolist() == g["inclusive"]
    assert gpu_segscan(ds, x, h, "add", False).tolist() == g["exclusive"]
    assert gpu_segscan(ds, x, h, "max", True).tolist() == g["max_inclusive"]


def test_segscan_f32_long_segments(ds):
    """fp32 add over segments far longer than a tile: the carry chain of
    tile aggregates is where the rounding accumulates."""
    rng = np.random.default_rng(54)
    n = 1 << 22
    x = rng.random(n, dtype=np.float32)
    h = np.zeros(n, np.uint8)
    h[[0, 12_345, 1_000_000, 3_000_001]] = 1
    for inclusive in (True, False):
        check(ds, x, h, "add", inclusive)
    assert F32_RTOL == 1e-5


def test_config_segmented(ds):
    from stream_compaction_device_gb300 import workloads as wl
    x, h = wl.segmented()
    for inclusive in (True, False):
        got = gpu_segscan(ds, x, h, "add", inclusive)
        ref = oracle.segscan(x, h, "add", inclusive)
        assert np.array_equal(got, ref)
        del got, ref
    assert ds.device_status() == 0
