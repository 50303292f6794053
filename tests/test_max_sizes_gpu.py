"""Maximum sizes, through the C ABI: scans of more than 2^32 elements (64-bit
element indexing, tile counts above 2^19) and compaction, the split and both
sorts at n = INT32_MAX, the largest count an int32 holds.

At these sizes a host copy of every array would take tens of GB, so each
result is checked on the device against the properties that define it, at
every element:
  * exclusive scan (geek-doc.cn "并行前缀和 scan ..." section 一): z[0] is the
    identity and z[i+1] = z[i] (+) x[i]; inclusive y = z (+) x;
  * compaction: the kept values in input order, i.e. values[flags != 0];
  * split: the keys whose bit is 0, in order, then those whose bit is 1;
  * sort: non-decreasing as uint32, and the same multiset as the input
    (three wrapping 64-bit sums of functions of the keys agree);
plus the first 2^20 elements of every scan against the serial oracle.
Inputs are drawn on the device with a seeded torch generator; torch only
evaluates the properties, never the operation itself.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

INT32_MAX = 2**31 - 1
HEAD = 1 << 20


@pytest.fixture(scope="module")
def ds():
    import stream_compaction_device_gb300 as m
    m.load()
    return m


def _gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("op", ["add", "max", "xor"])
def test_scan_beyond_2_to_32_elements(ds, op):
    n = (1 << 32) + 3
    lo, hi = (-3, 4) if op == "add" else (-2**31, 2**31 - 1)
    x = torch.randint(lo, hi, (n,), dtype=torch.int32, device="cuda", generator=_gen(11))
    z = ds.scan_exclusive(x, op=op)
    combine = {"add": torch.add, "max": torch.maximum, "xor": torch.bitwise_xor}[op]
    ident = {"add": 0, "max": -2**31, "xor": 0}[op]
    assert int(z[0].item()) == ident
    assert torch.equal(z[1:], combine(z[:-1], x[:-1])), "z[i+1] != z[i] op x[i] somewhere"
    head = x[:HEAD].cpu().numpy()
    assert np.array_equal(z[:HEAD].cpu().numpy(), oracle.scan(head, op, False))
    del z
    _free()
    y = ds.scan_inclusive(x, op=op)
    assert int(y[0].item()) == int(x[0].item())
    assert torch.equal(y[1:], combine(y[:-1], x[1:])), "y[i+1] != y[i] op x[i+1] somewhere"
    assert np.array_equal(y[:HEAD].cpu().numpy(), oracle.scan(head, op, True))
    assert ds.device_status() == 0
    del x, y
    _free()


def test_compaction_at_int32_max(ds):
    n = INT32_MAX
    v = torch.randint(-2**31, 2**31 - 1, (n,), dtype=torch.int32, device="cuda", generator=_gen(12))
    t = -1   # half kept
    want = v[v > t]
    flags = (v > t).to(torch.uint8)
    out, cnt = ds.compact(v, flags)
    k = int(cnt.item())
    assert k == want.numel()
    assert torch.equal(out[:k], want)
    del flags, out, cnt
    _free()
    out, cnt = ds.compact_greater(v, t)
    assert int(cnt.item()) == want.numel()
    assert torch.equal(out[:want.numel()], want)
    assert ds.device_status() == 0
    del v, want, out, cnt
    _free()


def test_compaction_keeps_everything_at_int32_max(ds):
    n = INT32_MAX
    v = torch.arange(n, dtype=torch.int32, device="cuda")
    out, cnt = ds.compact(v, torch.ones(n, dtype=torch.uint8, device="cuda"))
    assert int(cnt.item()) == INT32_MAX
    assert torch.equal(out, v)
    del v, out, cnt
    _free()


def test_split_at_int32_max(ds):
    n = INT32_MAX
    k = torch.randint(-2**31, 2**31 - 1, (n,), dtype=torch.int32, device="cuda", generator=_gen(13))
    bit = 13
    out = ds.split_bit(k, bit)
    one = ((k >> bit) & 1).bool()
    z = int((~one).sum().item())
    assert torch.equal(out[:z], k[~one])
    assert torch.equal(out[z:], k[one])
    assert ds.device_status() == 0
    del k, out, one
    _free()


def _multiset_hashes(keys: torch.Tensor):
    u = keys.to(torch.int64) & 0xFFFFFFFF
    return (int(u.sum().item()), int((u * u).sum().item()),
            int(((u * -7046029254386353131) ^ (u >> 7)).sum().item()))


@pytest.mark.parametrize("which", ["32pass", "digits"])
def test_sorts_at_int32_max(ds, which):
    n = INT32_MAX
    keys = torch.randint(-2**31, 2**31 - 1, (n,), dtype=torch.int32, device="cuda", generator=_gen(14))
    before = _multiset_hashes(keys)
    (ds.radix_sort if which == "32pass" else ds.radix_sort_digits)(keys)
    assert ds.device_status() == 0
    assert _multiset_hashes(keys) == before, "not a permutation of the input"
    u = keys.to(torch.int64) & 0xFFFFFFFF
    assert bool((u[1:] >= u[:-1]).all()), "not non-decreasing as uint32"
    del keys, u
    _free()
