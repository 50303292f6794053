"""Compaction, one-bit split and radix-sort parity: the CUDA library against
the CPU oracle, bit-exact, on seeded inputs from tiny and ragged sizes up to
the full workloads (N = 2^26)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import from_dev, to_dev

pytestmark = pytest.mark.gpu

TILE = 4096
SIZES = [1, 2, 3, 5, 15, 16, 17, 31, 32, 33, 127, 128, 129, 1023, 1024, 1025, TILE - 1, TILE, TILE + 1,
         8191, 8192, 8193, 3 * 8192 + 5, 65_536, 65_537, 300_007, 524_288, 524_291]


@pytest.fixture(scope="module")
def ds():
    import stream_compaction_device_gb300 as m
    m.load()
    return m


@pytest.fixture(params=["lookback", "pipelined", "l2"])
def mode(request, ds):
    """Run a test once on each kernel family (one tile per block; the
    persistent two-pass pipeline; for compaction in mode "l2", the two-launch
    count-then-write path at every size)."""
    ds.set_carry_mode(request.param)
    yield request.param
    ds.set_carry_mode("default")


def gpu_compact(ds, v: np.ndarray, f: np.ndarray, voff=0, foff=0, ooff=0):
    dv = to_dev(np.concatenate([np.zeros(voff, np.int32), v]))[voff:]
    df = torch.from_numpy(np.concatenate([np.zeros(foff, np.uint8), f])).cuda()[foff:]
    out = torch.full((v.size + ooff + 8,), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ds.compact(dv, df, out=out[ooff:ooff + max(v.size, 1)], count=cnt)
    torch.cuda.synchronize()
    k = int(cnt.item())
    host = out.cpu().numpy()
    # nothing written outside the kept range (guard words stay -7)
    assert np.all(host[:ooff] == -7) and np.all(host[ooff + k:] == -7)
    return host[ooff:ooff + k]


def check_compact(ds, v, f, **kw):
    got = gpu_compact(ds, v, f, **kw)
    ref = oracle.compact(v, f)
    assert got.size == ref.size, f"count {got.size} != {ref.size} (n={v.size})"
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"n={v.size}: first mismatch at {bad[0]}"


@pytest.mark.parametrize("pattern", ["random", "none", "all", "alternate", "sparse", "runs"])
def test_compact_sizes(ds, mode, pattern):
    rng = np.random.default_rng(21)
    for n in SIZES:
        v = rng.integers(-2**31, 2**31, n, dtype=np.int32)
        if pattern == "random":
            f = rng.integers(0, 4, n).astype(np.uint8)     # 1, 2, 3 all keep
        elif pattern == "none":
            f = np.zeros(n, np.uint8)
        elif pattern == "all":
            f = np.full(n, 255, np.uint8)
        elif pattern == "alternate":
            f = (np.arange(n) % 2).astype(np.uint8)
        elif pattern == "sparse":
            f = (rng.random(n) < 0.001).astype(np.uint8)
        else:
            f = ((np.arange(n) // 1000) % 2).astype(np.uint8)
        check_compact(ds, v, f)


@pytest.mark.parametrize("pattern", ["random2pct", "clustered", "mixed", "at_limit", "over_limit"])
def test_compact_sparse_tiles(ds, mode, pattern):
    """Tiles of 8,192 with few kept elements (256 or 257 each), tiles whose
    kept elements crowd one 512-element part, and sparse tiles next to dense
    ones."""
    rng = np.random.default_rng(sum(map(ord, pattern)))
    for n in (64 * 8192, 64 * 8192 + 4101, 1 << 21):
        v = rng.integers(-2**31, 2**31, n, dtype=np.int32)
        i = np.arange(n)
        if pattern == "random2pct":
            f = (rng.random(n) < 0.02).astype(np.uint8)
        elif pattern == "clustered":          # 200 kept, all in the tile's first part
            f = ((i % 8192) < 200).astype(np.uint8)
        elif pattern == "mixed":              # even tiles 1% kept, odd tiles 60%
            p = np.where((i // 8192) % 2 == 0, 0.01, 0.60)
            f = (rng.random(n) < p).astype(np.uint8)
        elif pattern == "at_limit":           # exactly 256 kept per tile
            f = ((i % 32) == 5).astype(np.uint8) * 9
        else:                                 # 257 kept per tile
            f = (((i % 32) == 5) | ((i % 8192) == 6)).astype(np.uint8)
        check_compact(ds, v, f)


@pytest.mark.parametrize("voff,foff,ooff", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (2, 3, 3), (0, 4, 2)])
def test_compact_unaligned(ds, mode, voff, foff, ooff):
    rng = np.random.default_rng(voff * 100 + foff * 10 + ooff)
    for n in (1, 77, TILE + 3, 200_001):
        v = rng.integers(-2**31, 2**31, n, dtype=np.int32)
        f = rng.integers(0, 2, n).astype(np.uint8)
        check_compact(ds, v, f, voff=voff, foff=foff, ooff=ooff)


def test_compact_empty(ds):
    v = torch.empty(0, dtype=torch.int32, device="cuda")
    f = torch.empty(0, dtype=torch.uint8, device="cuda")
    cnt = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    ds.compact(v, f, out=torch.empty(1, dtype=torch.int32, device="cuda"), count=cnt)
    assert int(cnt.item()) == 0


def test_compact_worked_example(ds, golden):
    g = golden("worked_example.txt")
    x = np.array(g["x"], dtype=np.int32)
    flags = (x > g["predicate_threshold"][0]).astype(np.uint8)
    assert gpu_compact(ds, x, flags).tolist() == g["compacted"]


@pytest.mark.parametrize("sel", [0.01, 0.50, 0.99])
def test_config_compaction(ds, sel):
    from stream_compaction_device_gb300 import workloads as wl
    v = wl.compaction_values()
    f = wl.predicate_flags(v, wl.threshold_for(sel))
    check_compact(ds, v, f)


# ---------------------------------------------------------------------------
# split and sort
# ---------------------------------------------------------------------------
def gpu_split(ds, k: np.ndarray, bit: int, koff=0, ooff=0):
    dk = to_dev(np.concatenate([np.zeros(koff, np.uint32), k]))[koff:]
    out = torch.full((k.size + ooff,), 0, dtype=torch.int32, device="cuda")
    ds.split_bit(dk, bit, out=out[ooff:])
    torch.cuda.synchronize()
    return from_dev(out, np.uint32)[ooff:]


@pytest.mark.parametrize("bit", [0, 1, 5, 16, 30, 31])
def test_split_sizes(ds, mode, bit):
    rng = np.random.default_rng(bit)
    for n in SIZES:
        k = rng.integers(0, 2**32, n, dtype=np.uint32)
        got = gpu_split(ds, k, bit)
        ref, _ = oracle.split_bit(k, bit)
        assert np.array_equal(got, ref), f"n={n} bit={bit}"


def test_split_skewed(ds, mode):
    rng = np.random.default_rng(3)
    for n in (TILE + 1, 100_003):
        for frac in (0.0, 0.001, 0.999, 1.0):
            k = rng.integers(0, 2**31, n, dtype=np.uint32)
            k[rng.random(n) < frac] |= np.uint32(1 << 31)
            assert np.array_equal(gpu_split(ds, k, 31), oracle.split_bit(k, 31)[0])


@pytest.mark.parametrize("koff,ooff", [(1, 0), (0, 1), (3, 2)])
def test_split_unaligned(ds, mode, koff, ooff):
    rng = np.random.default_rng(koff + 7 * ooff)
    for n in (1, 99, TILE + 5, 70_001):
        k = rng.integers(0, 2**32, n, dtype=np.uint32)
        assert np.array_equal(gpu_split(ds, k, 9, koff, ooff), oracle.split_bit(k, 9)[0])


def gpu_sort(ds, k: np.ndarray):
    d = to_dev(k)
    ds.radix_sort(d)
    torch.cuda.synchronize()
    return from_dev(d, np.uint32)


def test_sort_sizes(ds, mode):
    rng = np.random.default_rng(5)
    for n in (1, 2, 3, 100, TILE, TILE + 1, 65_537, 1_000_003):
        k = rng.integers(0, 2**32, n, dtype=np.uint32)
        k[: min(n, 6)] = np.array([0, 2**32 - 1, 7, 7, 2**31, 2**31 - 1], dtype=np.uint32)[: min(n, 6)]
        got = gpu_sort(ds, k)
        assert np.array_equal(got, oracle.sort_lsd(k)), f"n={n}"


def test_config_split_bits(ds):
    from stream_compaction_device_gb300 import workloads as wl
    k = wl.radix_keys()
    for bit in (0, 13, 31):
        assert np.array_equal(gpu_split(ds, k, bit), oracle.split_bit(k, bit)[0]), bit


def test_config_sort(ds):
    from stream_compaction_device_gb300 import workloads as wl
    k = wl.radix_keys()
    got = gpu_sort(ds, k)
    assert np.array_equal(got, np.sort(k))
    sample = k[: 1 << 20]
    assert np.array_equal(gpu_sort(ds, sample), oracle.sort_lsd(sample))
    assert ds.device_status() == 0


# ---------------------------------------------------------------------------
# 4-bit-digit radix sort
# ---------------------------------------------------------------------------
def gpu_sort_digits(ds, k: np.ndarray, koff=0):
    d = to_dev(np.concatenate([np.zeros(koff, np.uint32), k]))[koff:]
    ds.radix_sort_digits(d)
    torch.cuda.synchronize()
    return from_dev(d, np.uint32)


def test_sort_digits_sizes(ds):
    rng = np.random.default_rng(9)
    # around a warp's 1,024 keys and the 8,192-key tile of the scatter
    for n in (1, 2, 3, 15, 16, 17, 100, 1023, 1024, 1025, 4095, 4096, 4097, 8191, 8192, 8193, 8192 + 1025,
              2 * 8192 + 7000, 65_537, 1_000_003):
        k = rng.integers(0, 2**32, n, dtype=np.uint32)
        k[: min(n, 6)] = np.array([0, 2**32 - 1, 7, 7, 2**31, 2**31 - 1], dtype=np.uint32)[: min(n, 6)]
        assert np.array_equal(gpu_sort_digits(ds, k), oracle.sort_lsd(k)), f"n={n}"


def test_sort_digits_patterns(ds):
    rng = np.random.default_rng(10)
    n = 300_001
    cases = {
        "all equal": np.full(n, 0xDEADBEEF, np.uint32),
        "one digit": (rng.integers(0, 16, n) << 12).astype(np.uint32),
        "descending": np.arange(n, dtype=np.uint32)[::-1].copy(),
        "few values": rng.choice(np.array([3, 2**31, 5, 2**32 - 1], dtype=np.uint32), n),
    }
    for name, k in cases.items():
        assert np.array_equal(gpu_sort_digits(ds, k), np.sort(k)), name
    # unaligned keys (scalar load path)
    k = rng.integers(0, 2**32, 77_777, dtype=np.uint32)
    assert np.array_equal(gpu_sort_digits(ds, k, koff=1), np.sort(k))


def test_config_sort_digits(ds):
    from stream_compaction_device_gb300 import workloads as wl
    k = wl.radix_keys()
    assert np.array_equal(gpu_sort_digits(ds, k), np.sort(k))
    assert ds.device_status() == 0


def test_mixed_calls_one_stream(ds):
    """The two-launch compaction and split, the L2-resident scan and the
    read-only bracket check share one arrival counter in the stream's device
    state (last-block carries and grid barriers); interleaved on one stream,
    every call still gives the oracle's result."""
    from stream_compaction_device_gb300 import workloads as wl
    rng = np.random.default_rng(77)
    nc, n = (1 << 23) + 5, (1 << 21) + 5
    v = rng.integers(-2**31, 2**31, nc, dtype=np.int32)
    f = (rng.random(nc) < 0.3).astype(np.uint8)
    k = rng.integers(0, 2**32, n, dtype=np.uint32)
    x = wl.random_input(np.int32, n, 4, "add")
    w = (2 * rng.integers(0, 2, n) - 1).astype(np.int32)
    ref_c, ref_s, ref_x = oracle.compact(v, f), oracle.split_bit(k, 7)[0], oracle.scan(x, "add", False)
    ref_w = oracle.scan(w, "add", True)
    ref_neg, ref_final = int(ref_w.min() < 0), int(ref_w[-1])
    dv, df, dk, dx, dw = to_dev(v), torch.from_numpy(f).cuda(), to_dev(k), to_dev(x), to_dev(w)
    out = torch.empty_like(dv)
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    so, xo = torch.empty_like(dk), torch.empty_like(dx)
    res = torch.empty(2, dtype=torch.int32, device="cuda")
    for _ in range(4):
        ds.compact(dv, df, out=out, count=cnt)
        ds.split_bit(dk, 7, out=so)
        ds.scan_exclusive(dx, xo)
        ds.bracket_scan(dw, result=res, store=False)
        ds.compact(dv, df, out=out, count=cnt)
        torch.cuda.synchronize()
        kk = int(cnt.item())
        assert kk == ref_c.size and np.array_equal(out[:kk].cpu().numpy(), ref_c)
        assert np.array_equal(from_dev(so, np.uint32), ref_s)
        assert np.array_equal(xo.cpu().numpy(), ref_x)
        assert res.cpu().tolist() == [ref_neg, ref_final]
    assert ds.device_status() == 0


def test_default_two_launch_boundaries(ds):
    """Around the default's switch to the two-launch split and sort (2^20
    keys) and to the two-launch compaction (2^23 elements), aligned and not."""
    ds.set_carry_mode("default")
    rng = np.random.default_rng(8)
    for n in ((1 << 20) - 1, 1 << 20, (1 << 20) + 3, (1 << 20) + 1023, (1 << 20) + 1025):   # 1,024-key parts
        k = rng.integers(0, 2**32, n, dtype=np.uint32)
        assert np.array_equal(gpu_split(ds, k, 23), oracle.split_bit(k, 23)[0]), n
        assert np.array_equal(gpu_split(ds, k, 0, koff=1, ooff=2), oracle.split_bit(k, 0)[0]), n
        assert np.array_equal(gpu_sort(ds, k), np.sort(k)), n
    for n in ((1 << 23) - 1, (1 << 23) + 1):
        v = rng.integers(-2**31, 2**31, n, dtype=np.int32)
        f = (rng.random(n) < 0.05).astype(np.uint8)
        check_compact(ds, v, f)
        check_compact(ds, v, f, ooff=1)
