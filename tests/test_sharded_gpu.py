"""The scan of an array split into contiguous shards, through the C ABI.

Each shard takes the library calls one rank of a multi-device scan makes
(geek-doc.cn "并行前缀和 scan ..." section 四 lifted from blocks to shards):
its total (reduce_T), the fold of the totals of the shards before it (reduce_T
over the gathered totals: the carry) and its scan from that carry
(scan_*_carry_T).  Here the P shards run one after another on one GPU; the
concatenated outputs must equal the oracle's scan of the whole array:
bit-exact for the integer operators and fp32 max, within
|err_i| <= 1e-5 * sum_{j<=i} |x_j| for fp32 add.  reduce_T and the carry
scans are also checked on their own against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_f32_within, from_dev, to_dev

pytestmark = pytest.mark.gpu

CASES = [(np.int32, "add"), (np.int32, "max"), (np.int32, "xor"), (np.uint32, "add"), (np.uint32, "max"),
         (np.uint32, "xor"), (np.float32, "add"), (np.float32, "max")]


@pytest.fixture(scope="module")
def ds():
    import stream_compaction_device_gb300 as m
    m.load()
    return m


def _check(got, want, absp, dtype, op, what):
    """absp: the running sum of |x| over what each output folds (fp32 add)."""
    if dtype == np.float32 and op == "add":
        assert_f32_within(got, want, absp, what)
    elif dtype == np.float32:
        assert np.array_equal(got.astype(np.float64), want), what
    else:
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, f"{what}: first mismatch at {bad[0]}"


def _dev(a, offset=0):
    """Device copy of `a` starting `offset` elements into its allocation."""
    if not offset:
        return to_dev(a)
    return to_dev(np.concatenate([np.zeros(offset, a.dtype), a]))[offset:]


@pytest.mark.parametrize("dtype,op", CASES, ids=lambda v: getattr(v, "__name__", v))
def test_reduce(ds, dtype, op):
    """reduce_T against the last element of the oracle's inclusive scan
    (the identity for an empty input), aligned and at offsets 1-3."""
    from stream_compaction_device_gb300 import workloads as wl
    for n in (0, 1, 2, 3, 5, 4095, 4096, 4097, 4096 * 152 + 3, 1_000_003, (1 << 22) + 3):
        for offset in (0, 1, 3):
            if n == 0 and offset:
                continue
            x = wl.random_input(dtype, n, n + offset, op)
            d = _dev(x, offset) if n else torch.empty(0, dtype=torch.float32 if dtype == np.float32 else torch.int32,
                                                     device="cuda")
            got = from_dev(ds.reduce(d, op, as_uint32=dtype == np.uint32), dtype)
            if n == 0:
                want = np.array([oracle.identity(op, dtype)], dtype=np.float64 if dtype == np.float32 else dtype)
                assert got.astype(want.dtype).tolist() == want.tolist()
                continue
            want = oracle.scan(x, op, True)[-1:]
            if dtype == np.float32 and op == "add":
                assert abs(float(got[0]) - float(want[0])) <= 1e-5 * float(oracle.abs_prefix(x)[-1]), (n, offset)
            else:
                _check(got, want, None, dtype, op, f"reduce n={n} offset={offset}")


# sizes that take each scan path: the cluster scan (<= 2^16), the one-tile
# kernel (2^16 .. 2^17), the L2-resident scan (2^17 .. 2^24), the pipeline
SIZES = (1, 5, 8193, 65_536, 70_001, 300_007, (1 << 22) + 5, (1 << 24) + 8)


@pytest.mark.parametrize("dtype,op", CASES, ids=lambda v: getattr(v, "__name__", v))
@pytest.mark.parametrize("inclusive", [True, False], ids=["incl", "excl"])
def test_carry_scan(ds, dtype, op, inclusive):
    """scan_*_carry_T(x, c) equals the oracle's scan of [c] + x without its
    first (inclusive) or last (exclusive) element."""
    from stream_compaction_device_gb300 import workloads as wl
    for n in SIZES:
        x = wl.random_input(dtype, n, n + 3, op)
        c = wl.random_input(dtype, 1, n + 4, op)
        whole = np.concatenate([c, x])
        incl = oracle.scan(whole, op, True)
        want = incl[1:] if inclusive else incl[:-1]
        fn = ds.scan_inclusive_carry if inclusive else ds.scan_exclusive_carry
        got = from_dev(fn(to_dev(x), to_dev(c), op=op, as_uint32=dtype == np.uint32), dtype)
        absp = oracle.abs_prefix(whole) if dtype == np.float32 else None
        _check(got, want, None if absp is None else (absp[1:] if inclusive else absp[:-1]), dtype, op,
               f"carry scan n={n}")


def test_carry_scan_null_carry_is_the_plain_scan(ds):
    from stream_compaction_device_gb300 import workloads as wl
    for n in (7, 100_001, (1 << 20) + 3):
        x = wl.random_input(np.int32, n, n, "add")
        got = from_dev(ds.scan_exclusive_carry(to_dev(x), None), np.int32)
        assert np.array_equal(got, oracle.scan(x, "add", False))


def test_carry_scan_on_every_carry_path(ds):
    """The carry seeds tile 0 on the one-tile, pipelined and L2-resident
    paths alike (measurement hook)."""
    from stream_compaction_device_gb300 import workloads as wl
    for mode in ("lookback", "pipelined", "l2", "rts"):
        ds.set_carry_mode(mode)
        try:
            for n in (5, 4097, 1_000_003):
                x = wl.random_input(np.int32, n, n, "add")
                c = np.array([123_456], dtype=np.int32)
                incl = oracle.scan(np.concatenate([c, x]), "add", True)
                got = from_dev(ds.scan_inclusive_carry(to_dev(x), to_dev(c)), np.int32)
                assert np.array_equal(got, incl[1:]), (mode, n)
        finally:
            ds.set_carry_mode("default")


def _sharded_sequential(ds, x, parts, op, inclusive, dtype):
    """Rank r's calls, for r = 0 .. P-1 in turn: the shard totals gathered
    into one device array, each shard's carry folded from those before it."""
    u32 = dtype == np.uint32
    shards = np.array_split(x, parts)
    d_shards, totals = [], []
    for s in shards:
        d = to_dev(s) if s.size else torch.empty(0, dtype=torch.float32 if dtype == np.float32 else torch.int32,
                                                device="cuda")
        d_shards.append(d)
        totals.append(ds.reduce(d, op, as_uint32=u32))
    gathered = torch.cat(totals)   # what the all-gather leaves on every device
    outs = []
    for r, d in enumerate(d_shards):
        carry = ds.reduce(gathered[:r], op, as_uint32=u32)
        fn = ds.scan_inclusive_carry if inclusive else ds.scan_exclusive_carry
        outs.append(from_dev(fn(d, carry, op=op, as_uint32=u32), dtype) if d.numel() else np.empty(0, dtype))
    return np.concatenate(outs)


@pytest.mark.parametrize("parts", [2, 3, 4])
@pytest.mark.parametrize("dtype,op", CASES, ids=lambda v: getattr(v, "__name__", v))
def test_sharded_scan_matches_whole_array(ds, parts, dtype, op):
    from stream_compaction_device_gb300 import workloads as wl
    for n in (parts - 1, 1_000_003, (1 << 24) + 13):
        x = wl.random_input(dtype, n, n + parts, op)
        for inclusive in (True, False):
            got = _sharded_sequential(ds, x, parts, op, inclusive, dtype)
            absp = oracle.abs_prefix(x) if dtype == np.float32 else None
            _check(got, oracle.scan(x, op, inclusive), absp, dtype, op, f"P={parts} n={n} incl={inclusive}")
    assert ds.device_status() == 0


def test_sharded_scan_full_size(ds):
    """The 2^28 bracket workload in 4 shards of 2^26 (the pipelined path with
    a carry), exclusive add, against the oracle's whole-array scan."""
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.brackets()
    got = _sharded_sequential(ds, x, 4, "add", False, np.int32)
    assert np.array_equal(got, oracle.scan(x, "add", False))


def test_sharded_scan_single_process(ds):
    """Without a process group the sharded scan is the whole scan."""
    from stream_compaction_device_gb300 import workloads as wl
    x = wl.random_input(np.int32, 300_001, 9, "add")
    got = from_dev(ds.sharded_scan(to_dev(x), inclusive=True), np.int32)
    assert np.array_equal(got, oracle.scan(x, "add", True))


def test_sharded_scan_through_a_one_rank_nccl_group(ds, tmp_path):
    """exchange_totals and sharded_scan through torch.distributed with NCCL
    (one rank: every call of this run has one GPU), against the oracle."""
    import torch.distributed as dist
    from stream_compaction_device_gb300 import workloads as wl
    dist.init_process_group("nccl", init_method=f"file://{tmp_path / 'store'}", rank=0, world_size=1)
    try:
        t = torch.tensor([42], dtype=torch.int32, device="cuda")
        assert ds.exchange_totals(t).tolist() == [42]
        for op in ("add", "max", "xor"):
            x = wl.random_input(np.int32, 1_000_003, 17, op)
            got = from_dev(ds.sharded_scan(to_dev(x), op=op), np.int32)
            assert np.array_equal(got, oracle.scan(x, op, False)), op
    finally:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# sharded compaction: each shard compacted, the counts folded into offsets
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("parts", [2, 3, 4])
@pytest.mark.parametrize("by_threshold", [True, False], ids=["predicate", "flags"])
@pytest.mark.parametrize("sel", [0.01, 0.5])
def test_sharded_compaction_matches_whole_array(ds, parts, by_threshold, sel):
    """P shards of one array, compacted one after another on one GPU through
    the calls one rank of sharded_compact makes: each shard's compaction,
    then the fold of the kept counts of the shards before it (its offset)
    and of all of them (the total).  The shards' kept values, placed at
    their offsets, are the oracle's compaction of the whole array."""
    from stream_compaction_device_gb300 import workloads as wl
    n = (1 << 22) + 12_345
    v = wl.compaction_values(n, seed=11)
    t = wl.threshold_for(sel)
    ref = oracle.compact(v, wl.predicate_flags(v, t))
    outs, counts = [], []
    for shard in np.array_split(v, parts):
        dv = to_dev(shard)
        if by_threshold:
            o, c = ds.compact_greater(dv, t)
        else:
            o, c = ds.compact(dv, torch.from_numpy(wl.predicate_flags(shard, t)).cuda())
        outs.append(o)
        counts.append(c)
    counts = torch.cat(counts)
    whole = np.empty(ref.size, np.int32)
    for r in range(parts):
        off = int(ds.reduce(counts[:r]).item())
        k = int(counts[r].item())
        assert off == int(counts[:r].sum().item())
        whole[off:off + k] = from_dev(outs[r][:k], np.int32)
    assert int(ds.reduce(counts).item()) == ref.size
    assert np.array_equal(whole, ref)
    assert ds.device_status() == 0


def test_sharded_compaction_single_process(ds):
    """Without a process group sharded_compact is the plain compaction:
    offset 0 and total = count."""
    from stream_compaction_device_gb300 import workloads as wl
    v = wl.compaction_values(1_000_003, seed=12)
    t = wl.threshold_for(0.2)
    ref = oracle.compact(v, wl.predicate_flags(v, t))
    out, cnt, off, tot = ds.sharded_compact(to_dev(v), threshold=t)
    assert (int(cnt.item()), int(off.item()), int(tot.item())) == (ref.size, 0, ref.size)
    assert np.array_equal(from_dev(out[: ref.size], np.int32), ref)
