"""The library's calls inside a CUDA graph: after one warm-up on the
capturing stream (which sets up that stream's workspace and scratch), a
capture of scans (cluster, L2-resident and pipelined sizes), the two-launch
compaction, the fused-predicate compaction (one cooperative launch that
captures or goes on as the pipeline, on inputs that keep 1% in one replay
and everything in the next), the standalone split, the 32-pass sort, the 8-bit digit sort and
one shard's calls of the sharded scan (its fold, the fold of the gathered
totals, its scan from that carry) replays with new inputs and matches the
CPU oracle each time.  The kernels keep their
look-back tags, tickets and arrival counters in device memory, so a replay
needs no host-side state."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ds():
    import stream_compaction_device_gb300 as m
    m.load()
    return m


def test_graph_capture_and_replay(ds):
    ds.set_carry_mode("default")
    rng = np.random.default_rng(2024)
    n_small, n_mid, n_big = 50_000, (1 << 21) + 3, (1 << 24) + 5
    nc, nk = (1 << 23) + 7, (1 << 20) + 5
    ng = (1 << 22) + 7

    def fresh():
        return {
            "xs": rng.integers(-1000, 1000, n_small, dtype=np.int32),
            "xm": rng.random(n_mid, dtype=np.float32),
            "xb": rng.integers(0, 2**32, n_big, dtype=np.uint32),
            "v": rng.integers(-2**31, 2**31, nc, dtype=np.int32),
            "f": (rng.random(nc) < 0.4).astype(np.uint8),
            "k": rng.integers(0, 2**32, nk, dtype=np.uint32),
            "g": rng.integers(-1000, 1000, ng, dtype=np.int32),   # about 1% above 979
        }

    h = fresh()
    xs, xm, xb = to_dev(h["xs"]), to_dev(h["xm"]), to_dev(h["xb"])
    v, f, k = to_dev(h["v"]), torch.from_numpy(h["f"]).cuda(), to_dev(h["k"])
    ys, ym, yb = torch.empty_like(xs), torch.empty_like(xm), torch.empty_like(xb)
    out, cnt = torch.empty_like(v), torch.empty(1, dtype=torch.int32, device="cuda")
    ko, work, tmp = torch.empty_like(k), torch.empty_like(k), torch.empty_like(k)
    work2 = torch.empty_like(k)
    gv = to_dev(h["g"])
    gout, gcnt = torch.empty_like(gv), torch.empty(1, dtype=torch.int32, device="cuda")
    totals = torch.empty(3, dtype=torch.int32, device="cuda")
    carry, ysh = torch.empty(1, dtype=torch.int32, device="cuda"), torch.empty_like(xs)

    def run():
        ds.scan_exclusive(xs, ys)                       # one thread-block cluster
        ds.scan_inclusive(xm, ym)                       # L2-resident cooperative scan
        ds.scan_inclusive(xb, yb, op="xor", as_uint32=True)   # the pipeline
        ds.compact(v, f, out=out, count=cnt)            # count launch, then write launch
        ds.compact_greater(gv, 979, out=gout, count=gcnt)   # cooperative: capture, or the pipeline
        ds.split_bit(k, 9, out=ko)
        work.copy_(k)
        ds.radix_sort(work, tmp)
        work2.copy_(k)
        ds.radix_sort_digits(work2, tmp)
        # shard 2 of 3 of an array whose other shards' totals sit in totals[0:2]
        ds.reduce(xs, out=totals[2:3])
        ds.reduce(totals[:2], out=carry)
        ds.scan_inclusive_carry(xs, carry, ysh)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    torch.cuda.synchronize()

    for rep in range(4):
        h = fresh()
        if rep % 2 == 1:   # everything kept: the capture gives up (then the stream backs off)
            h["g"] = rng.integers(980, 2000, ng, dtype=np.int32)
        for dst, src in ((xs, h["xs"]), (xm, h["xm"]), (xb, h["xb"]), (v, h["v"]), (k, h["k"]), (gv, h["g"])):
            dst.copy_(to_dev(src))
        f.copy_(torch.from_numpy(h["f"]).cuda())
        t01 = rng.integers(-10**6, 10**6, 2, dtype=np.int32)
        totals[:2].copy_(torch.from_numpy(t01).cuda())
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(ys.cpu().numpy(), oracle.scan(h["xs"], "add", False))
        ref_m = oracle.scan(h["xm"], "add", True)
        assert np.all(np.abs(ym.cpu().numpy().astype(np.float64) - ref_m)
                      <= 1e-5 * oracle.abs_prefix(h["xm"]))
        assert np.array_equal(from_dev(yb, np.uint32), oracle.scan(h["xb"], "xor", True))
        kk = int(cnt.item())
        ref_c = oracle.compact(h["v"], h["f"])
        assert kk == ref_c.size and np.array_equal(out[:kk].cpu().numpy(), ref_c)
        kg = int(gcnt.item())
        ref_g = h["g"][h["g"] > 979]
        assert kg == ref_g.size and np.array_equal(gout[:kg].cpu().numpy(), ref_g)
        assert np.array_equal(from_dev(ko, np.uint32), oracle.split_bit(h["k"], 9)[0])
        assert np.array_equal(from_dev(work, np.uint32), np.sort(h["k"]))
        assert np.array_equal(from_dev(work2, np.uint32), np.sort(h["k"]))
        assert int(totals[2].item()) == int(oracle.scan(h["xs"], "add", True)[-1])
        shard = oracle.scan(np.concatenate([t01, h["xs"]]), "add", True)[2:]
        assert np.array_equal(ysh.cpu().numpy(), shard)
    assert ds.device_status(s) == 0
    ds.stream_release(s)
