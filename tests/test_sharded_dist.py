"""The exchange step of the sharded scan, as gloo ranks on the CPU.

``exchange_totals`` gathers one total per rank into every rank's array in
rank order; ``sharded_scan`` folds the totals of the ranks before this one
into the carry.  The device calls (the shard's total, the fold of the
gathered totals and the carry scan) need a GPU, so here each rank replaces
them with host stand-ins built from the oracle, and the test checks only
the wiring between them: concatenated in rank order, the ranks' outputs
must be the oracle's scan of the whole array.  The library calls
themselves are checked on the GPU in test_sharded_gpu.py.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _host_stand_ins(ds, oracle):
    """Oracle-based replacements for the three device calls (test only)."""
    def reduce(x, op="add", out=None, stream=None, as_uint32=False):
        a = x.numpy()
        if a.size == 0:
            return torch.tensor([oracle.identity(op, a.dtype)], dtype=x.dtype)
        return torch.from_numpy(oracle.scan(a, op, True)[-1:].astype(a.dtype))

    def carry_scan(inclusive):
        def fn(x, carry, out=None, op="add", stream=None, as_uint32=False):
            a = x.numpy()
            incl = oracle.scan(np.concatenate([carry.numpy()[:1], a]), op, True)
            return torch.from_numpy((incl[1:] if inclusive else incl[:-1]).astype(a.dtype))
        return fn
    ds.reduce = reduce
    ds.scan_inclusive_carry = carry_scan(True)
    ds.scan_exclusive_carry = carry_scan(False)


def _worker(rank, world, port, n, op, inclusive, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import oracle
    import stream_compaction_device_gb300 as ds
    from stream_compaction_device_gb300 import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        totals = ds.exchange_totals(torch.tensor([10 * rank + 1], dtype=torch.int32))
        out[("totals", rank)] = totals.tolist()
        _host_stand_ins(ds, oracle)
        x = wl.random_input(np.int32, n, 5, op)
        shard = torch.from_numpy(np.array_split(x, world)[rank].copy())
        out[("scan", rank)] = ds.sharded_scan(shard, inclusive=inclusive, op=op).numpy().tolist()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,op,inclusive", [(2, "add", False), (2, "max", True), (3, "xor", False),
                                                (3, "add", True)])
def test_exchange_and_fold_wiring(world, op, inclusive):
    import oracle
    from stream_compaction_device_gb300 import workloads as wl
    n = 1_001
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, op, inclusive, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    for r in range(world):
        assert out[("totals", r)] == [10 * q + 1 for q in range(world)]
    got = np.concatenate([np.array(out[("scan", r)], dtype=np.int32) for r in range(world)])
    x = wl.random_input(np.int32, n, 5, op)
    assert np.array_equal(got, oracle.scan(x, op, inclusive))


def test_single_process_exchange_is_the_total():
    import stream_compaction_device_gb300 as ds
    t = torch.tensor([7], dtype=torch.int32)
    assert ds.exchange_totals(t).tolist() == [7]


# ---------------------------------------------------------------------------
# sharded compaction: the same exchange, with kept counts
# ---------------------------------------------------------------------------
def _compact_stand_ins(ds, oracle):
    """Oracle-based replacements for the device compaction and fold (test
    only)."""
    def compact(values, flags, out=None, count=None, stream=None):
        kept = oracle.compact(values.numpy(), flags.numpy())
        res = torch.zeros(values.numel(), dtype=torch.int32)
        res[: kept.size] = torch.from_numpy(kept.astype(np.int32))
        return res, torch.tensor([kept.size], dtype=torch.int32)

    def compact_greater(values, threshold, out=None, count=None, stream=None):
        v = values.numpy()
        return compact(values, torch.from_numpy((v > np.int32(threshold)).astype(np.uint8)))

    def reduce(x, op="add", out=None, stream=None, as_uint32=False):
        return torch.tensor([int(x.numpy().astype(np.int64).sum())], dtype=x.dtype)
    ds.compact = compact
    ds.compact_greater = compact_greater
    ds.reduce = reduce


def _compact_worker(rank, world, port, n, by_threshold, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import oracle
    import stream_compaction_device_gb300 as ds
    from stream_compaction_device_gb300 import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _compact_stand_ins(ds, oracle)
        v = wl.compaction_values(n, seed=9)
        t = wl.threshold_for(0.3)
        shard = torch.from_numpy(np.array_split(v, world)[rank].copy())
        if by_threshold:
            res, cnt, off, tot = ds.sharded_compact(shard, threshold=t)
        else:
            f = torch.from_numpy(wl.predicate_flags(shard.numpy(), t))
            res, cnt, off, tot = ds.sharded_compact(shard, flags=f)
        k = int(cnt.item())
        out[("kept", rank)] = res[:k].numpy().tolist()
        out[("place", rank)] = (int(off.item()), int(tot.item()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,by_threshold", [(2, True), (3, False), (4, True)])
def test_sharded_compaction_wiring(world, by_threshold):
    """Concatenated in rank order, the ranks' kept values are the oracle's
    compaction of the whole array; each rank's offset is the kept count of
    the ranks before it, and every rank gets the whole count."""
    import oracle
    from stream_compaction_device_gb300 import workloads as wl
    n = 10_007
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_compact_worker, args=(r, world, port, n, by_threshold, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    v = wl.compaction_values(n, seed=9)
    ref = oracle.compact(v, wl.predicate_flags(v, wl.threshold_for(0.3)))
    got = [np.array(out[("kept", r)], dtype=np.int32) for r in range(world)]
    assert np.array_equal(np.concatenate(got), ref)
    at = 0
    for r in range(world):
        assert out[("place", r)] == (at, ref.size)
        at += got[r].size
