"""Host logic of the multi-replica benchmark: with N ranks the reported time
is the maximum over ranks and the work is the sum over ranks (weak scaling,
independent replicas).  Runs as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, u = bench.aggregate(1.0 + rank, 100.0 * (rank + 1), world)
    out[rank] = (t, u)
    bench.barrier(world)
    dist.destroy_process_group()


def test_aggregate_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 300.0)


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_reference_arm_line(capsys):
    """The reference arm prints one JSON line with the oracle as baseline."""
    import json
    import bench
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1", "--n", str(1 << 23)])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "Gelem/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


@pytest.mark.gpu
@pytest.mark.parametrize("op", ["compact50", "segscan", "bracket_check", "split", "sort32", "digit_sort"])
def test_single_op_mode(capsys, op):
    """``bench.py --op``: one library call repeated for a profiler, its own line."""
    import json
    import bench
    bench.main(["--op", op, "--n", "300007", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["op"] == op and line["n"] == 300007 and line["status"] == 0 and line["ms_per_call"] > 0
