#!/usr/bin/env python3
"""Benchmark of the device-wide scan library on GB300.

One step = one int32 exclusive add-scan of N = 2^28 elements (the +1/-1
bracket sequence, seed 3) through the C ABI, inputs resident in HBM.  The
inputs (1 GiB in, 1 GiB out) are far larger than the 126 MB L2, so no flush
is needed between steps.  Prints one JSON line:

  value      whole-job Gelem/s (all ranks' elements / max-over-ranks time)
  roofline   the scan kernel's algorithmic bytes (2 * N * 4 per launch) over
             its CUDA-event duration, against the measured HBM copy peak
  e2e        the same scan from pinned host memory through the library's
             host entry (scan_exclusive_host_i32: host-to-device copy, scan,
             device-to-host copy of the result, all queued by the library),
             every step; steps alternate between two streams, so one step's
             download overlaps the next one's upload
  cpu_baseline  the serial CPU oracle on the host cores (1 thread)
  cpu_baseline_mt  the blocked three-phase scan on every host core
  extra      the inclusive / max / xor sweep, the bracket check and bracket
             scan, the segmented scan, the fold and one rank's share of the
             sharded scan at N = 2^28; compaction (flags; fused predicate
             by default, two-launch and pipelined alone), the split, the
             32-pass and the 8-bit radix
             sorts at N = 2^26; fp32 add at N = 2^24; N = 65,536 latency; the
             reduce-then-scan carry.  Back-to-back calls between one pair of
             events (device time per call), except the rows that flush L2
             (a read of 256 MiB before each call; per-call events, 10%-trimmed
             mean of at least 200 calls)

``--impl reference`` times the CPU oracle instead (the reference arm): each
step is the oracle's serial exclusive scan of the same 2^28-element
workload, on one host core.  With ``--gpus N`` > 1 (launched by torchrun) every rank runs
an independent replica on its own GPU (the scan needs no exchange between
replicas); ``scaling`` is "weak".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "int32 exclusive scan Gelem/s & HBM GB/s (% peak) at N=2^28; compaction Gelem/s"
N_HEADLINE = 1 << 28
REF_FULL_STEPS = 600   # whole-array oracle scans the reference arm may run (about 130 s at 2^28)
FALLBACK_HBM_GBS = 6800.0
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the pipelined
# scan kernel at N = 2^28 (one-pass ncu capture of this benchmark's own
# command); set to None whenever the kernel changes until it is re-captured.
SCAN_TRAFFIC_BYTES = 2.147e9


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def aggregate(elapsed_s: float, units: float, world: int, device=None):
    """Max of the elapsed times and sum of the units over all ranks."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class _Nvml:
    """The few NVML queries the clock record needs, through ctypes (the GPU
    hosts have the driver's libnvidia-ml but not every Python wrapper).
    Reads only: no setting of the GPU is changed."""
    SM_CLOCK = 1   # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        uuid = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
        except Exception:
            pass
        rc = 1
        if uuid:
            rc = self.lib.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(self.dev))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.dev))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.SM_CLOCK)

    def cpu_affinity(self):
        """The host CPUs NVML names as closest to the device (a set), or
        None when the query is unavailable."""
        words = 64
        mask = (self.c.c_ulong * words)()
        if self.lib.nvmlDeviceGetCpuAffinity(self.dev, words, mask) != 0:
            return None
        bits = self.c.sizeof(self.c.c_ulong) * 8
        return {w * bits + b for w in range(words) for b in range(bits) if (mask[w] >> b) & 1}

    def _uint(self, fn, *args):
        v = self.c.c_uint()
        return v.value if fn(self.dev, *args, self.c.byref(v)) == 0 else None

    def sample(self):
        r = self.c.c_ulonglong()
        reasons = r.value if self.reasons_fn(self.dev, self.c.byref(r)) == 0 else 0
        mw = self._uint(self.lib.nvmlDeviceGetPowerUsage)
        return (time.perf_counter(), self._uint(self.lib.nvmlDeviceGetClockInfo, self.SM_CLOCK), self.max_mhz,
                None if mw is None else mw / 1e3, sorted(n for bit, n in self.REASONS.items() if reasons & bit))


class HostPlacement:
    """Binds the calling thread to the host CPUs closest to GPU ``index``
    (those NVML names, within the CPUs this process may use) until
    ``restore``; ``info`` records what was found and done."""

    def __init__(self, index: int):
        self.saved = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
        self.info = {"bound": False}
        try:
            near = _Nvml(index).cpu_affinity()
        except Exception as exc:   # no NVML on this host: leave the placement alone
            self.info["why"] = f"no NVML CPU affinity ({type(exc).__name__})"
            return
        if not near or self.saved is None:
            self.info["why"] = "NVML gave no CPU affinity"
            return
        use = self.saved & near
        self.info.update({"allowed_cpus": len(self.saved), "gpu_near_cpus": len(near), "both": len(use)})
        if not use:
            self.info["why"] = "none of this process's CPUs is near the GPU"
            return
        os.sched_setaffinity(0, use)
        self.info["bound"] = True

    def restore(self):
        if self.saved is not None and self.info.get("bound"):
            os.sched_setaffinity(0, self.saved)


class ClockSampler:
    """SM clock, power and throttle reasons sampled every ``period_s`` on a
    background thread while the timed region runs (NVML through ctypes; the
    bench's timed regions last milliseconds, below nvidia-smi's polling
    interval).  ``stop`` summarises the samples taken between the marks t0
    and t1; with none inside, ``sm_mhz`` is null and ``why_null`` says so."""

    def __init__(self, gpu_index: int, period_s: float = 0.0005):
        self.gpu = gpu_index
        self.period = period_s
        self.samples = []
        self.t0 = self.t1 = None
        self.thread = None
        self.error = None

    def start(self):
        import threading
        try:
            self.nvml = _Nvml(self.gpu)
        except (OSError, AttributeError) as e:
            self.error = f"NVML unavailable: {e}"
            return
        self.halt = threading.Event()

        def run():
            while not self.halt.is_set():
                self.samples.append(self.nvml.sample())
                time.sleep(self.period)
        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()
        time.sleep(0.05)

    def mark(self, which):
        setattr(self, which, time.perf_counter())

    def stop(self):
        if self.thread is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "why_null": self.error or "sampler not started"}
        self.halt.set()
        self.thread.join(5)
        inside = [s for s in self.samples if self.t0 is not None and self.t1 is not None and self.t0 <= s[0] <= self.t1]
        out = {"samples": len(self.samples), "samples_in_timed_region": len(inside), "source": "nvml",
               "period_ms": self.period * 1e3,
               "timed_region_ms": None if self.t0 is None or self.t1 is None else round((self.t1 - self.t0) * 1e3, 3)}
        if not inside:
            out.update(sm_mhz=None, sm_max_mhz=self.nvml.max_mhz, reasons=[],
                       why_null="no clock sample fell inside the timed region")
            return out
        mhz = [s[1] for s in inside if s[1] is not None]
        out.update(sm_mhz=statistics.median(mhz) if mhz else None, sm_min_mhz=min(mhz) if mhz else None,
                   sm_max_mhz=self.nvml.max_mhz, reasons=sorted({r for s in inside for r in s[4]}),
                   power_w_max=max((s[3] for s in inside if s[3] is not None), default=None))
        return out


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------
def time_events(fn, reps, warmup, flush=None):
    """Per-call milliseconds of fn() with CUDA events on the current stream,
    as (median, mean; with ``flush``: the 10%-trimmed mean).  Without ``flush`` the calls run back to back between
    one pair of events, as the headline steps do, so the host's launch
    overhead overlaps the device work and the result is the device time per
    call (median and mean are then the same number).  With ``flush`` (run
    between calls, outside the events) every call gets its own pair of events;
    everything is enqueued before the one synchronize at the end, so the
    device never waits on the host inside a pair."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if flush is None:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        b.synchronize()
        per = a.elapsed_time(b) / reps
        return per, per
    pairs = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        pairs.append((a, b))
    torch.cuda.synchronize()
    times = sorted(a.elapsed_time(b) for a, b in pairs)
    k = len(times) // 10   # the 10%-trimmed mean: the event timer ticks in steps of about 2 us, so a
    return statistics.median(times), statistics.fmean(times[k:len(times) - k])   # single median snaps to a tick


def cpu_mt_rate(x: np.ndarray, budget_s: float):
    """Multithreaded CPU baseline (blocked three-phase scan on every host
    core) throughput in Gelem/s, repeated until ``budget_s`` seconds pass;
    returns (rate, runs, seconds, threads used)."""
    import oracle
    _, used = oracle.mt_scan_exclusive_add(x[:1 << 16])
    reps, t0 = 0, time.perf_counter()
    while True:
        _, used = oracle.mt_scan_exclusive_add(x)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s and reps >= 2:
            break
    return x.size * reps / el / 1e9, reps, el, used


def cpu_oracle_rate(x: np.ndarray, budget_s: float):
    """Serial oracle exclusive add-scan throughput (Gelem/s) on repeated runs
    over ``x`` until ``budget_s`` seconds of CPU work have been spent."""
    import oracle
    oracle.scan(x[:1024], "add", False)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.scan(x, "add", False)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s and reps >= 2:
            break
    return x.size * reps / el / 1e9, reps, el


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    import stream_compaction_device_gb300 as ds
    from stream_compaction_device_gb300 import workloads as wl

    ds.load()
    if args.carry != "default":
        ds.set_carry_mode(args.carry)
    n = args.n
    peak, peak_kind = peak_hbm()
    x_host = wl.brackets(n)
    d_in = torch.from_numpy(x_host).cuda()
    d_out = torch.empty_like(d_in)
    stream = torch.cuda.current_stream()
    launches_per_step = 3 if args.carry == "rts" else 1

    def step():
        ds.scan_exclusive(d_in, d_out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if rank == 0 and not args.no_clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("t0")
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    barrier(world)
    elapsed = ev0.elapsed_time(ev1) / 1e3
    assert ds.device_status() == 0, "device-side error during the timed region"
    t_max, units = aggregate(elapsed, float(n) * args.steps, world, torch.device("cuda", local))
    clock_info = clocks.stop() if (rank == 0 and not args.no_clocks) else None

    # parity spot check of the timed output (last step) against the oracle
    # on sampled positions: z[i] = sum of x[0..i-1]
    idx = np.unique(np.concatenate([np.arange(8), np.random.default_rng(0).integers(0, n, 64), [n - 1]]))
    pref = np.concatenate([[0], np.cumsum(x_host, dtype=np.int64)])
    got = d_out[torch.from_numpy(idx).cuda()].cpu().numpy()
    parity_ok = bool(np.array_equal(got.astype(np.int64), pref[idx]))

    value = units / t_max / 1e9
    kernel_s = elapsed / args.steps
    alg_bytes = 2 * n * 4
    achieved = alg_bytes / kernel_s / 1e9

    # end to end from pinned host memory through the public API
    e2e = None
    if not args.no_e2e:
        # steps alternate between two streams (each with its own device and
        # pinned output buffers), so one step's download overlaps the next
        # step's upload, as a user streaming batches would run it; every step
        # still moves its whole input up and its whole result down
        # the pinned buffers are first touched from the CPUs closest to the
        # GPU, so that their pages sit on the GPU's side of the host (a
        # buffer on the far socket crosses the socket link on every copy)
        placement = HostPlacement(local)
        h_in = torch.from_numpy(x_host).pin_memory()
        h_outs = [torch.empty_like(h_in).pin_memory() for _ in range(2)]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        works = [(d_in, d_out), (torch.empty_like(d_in), torch.empty_like(d_out))]
        e2e_steps = max(4, min(20, args.steps))
        for j in range(2):
            ds.scan_host(h_in, inclusive=False, out_host=h_outs[j], work=works[j], stream=streams[j])
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            j = i % 2
            ds.scan_host(h_in, inclusive=False, out_host=h_outs[j], work=works[j], stream=streams[j],
                         synchronize=False)
        torch.cuda.synchronize()
        el = time.perf_counter() - t0
        el, u = aggregate(el, float(n) * e2e_steps, world, torch.device("cuda", local))
        e2e = {"value": round(u / el / 1e9, 3), "unit": "Gelem/s", "h2d_bytes_per_step": n * 4,
               "d2h_bytes_per_step": n * 4, "steps": e2e_steps, "host_placement": placement.info}
        del h_in, h_outs, works
        placement.restore()

    extra = None
    if not args.no_extras and rank == 0:
        extra = run_extras(args, ds, wl, d_in, d_out, peak)

    cpu = cpu_mt = None
    if rank == 0 and world >= 1 and not args.no_cpu:
        rate, reps, el = cpu_oracle_rate(x_host, args.cpu_budget)
        cpu = {"value": round(rate, 4), "unit": "Gelem/s", "cores": 1, "kind": "oracle",
               "sample": f"serial oracle exclusive add-scan of the full 2^{n.bit_length() - 1}-element "
                         f"workload, {reps} runs, {el:.1f} s"}
        rate, reps, el, used = cpu_mt_rate(x_host, args.cpu_budget / 2)
        cpu_mt = {"value": round(rate, 4), "unit": "Gelem/s", "cores": used, "kind": "blocked three-phase, threads",
                  "sample": f"multithreaded blocked exclusive add-scan of the full 2^{n.bit_length() - 1}-element "
                            f"workload on {used} host threads, {reps} runs, {el:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "Gelem/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_max / args.steps * 1e3, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic",
            "config": {"workload": f"int32 exclusive add-scan, N=2^{n.bit_length() - 1}, +1/-1 bracket "
                                   "sequence (p=0.5, seed 3)", "n": n, "op": "add", "inclusive": False,
                       "carry": args.carry, "tile_elems": 8192,
                       "l2": "input and output 1 GiB each (> 126 MB L2); no flush between steps",
                       "replicas": world},
            "hbm_gbs": round(achieved, 1), "pct_peak": round(100 * achieved / peak, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": SCAN_TRAFFIC_BYTES,
                         "kernel": "pipeline_l2_kernel<ScanPolicy<AddU32,exclusive,16,4,4,2,4,10,prefetch 1,parts,2 tiles per ticket>>",
                         "algorithmic_bytes_per_launch": alg_bytes, "peak_kind": peak_kind},
            "cpu_baseline": cpu, "cpu_baseline_mt": cpu_mt, "e2e": e2e, "gpu_launches": args.steps * launches_per_step,
            "clocks": clock_info, "parity_sampled": parity_ok, "extra": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_extras(args, ds, wl, d_in, d_out, peak):
    """Secondary rows, timed with CUDA events: back-to-back calls between one
    event pair (device time per call), except the rows that flush L2 between
    calls, which are timed call by call."""
    import torch
    out = {}
    reps = args.extra_reps
    # L2 flush between calls of the rows that fit in L2: a read of 256 MiB (a
    # sum into one scalar) replaces every line with a clean one, so no
    # write-back of dirty lines lands inside the next timed call
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    flush_acc = torch.empty((), dtype=torch.float32, device="cuda")

    def flush():
        torch.sum(flush_buf, dim=0, out=flush_acc)

    def row(n_elems, ms, nbytes):
        gbs = nbytes / (ms / 1e3) / 1e9
        return {"us": round(ms * 1e3, 2), "gelem_s": round(n_elems / (ms / 1e3) / 1e9, 2),
                "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}

    n = d_in.numel()
    # inclusive add on the same array, and the max / xor sweep
    med, _ = time_events(lambda: ds.scan_inclusive(d_in, d_out), reps, 3)
    out["i32_add_inclusive_2^28"] = row(n, med, 8 * n)
    # the bracket check on the same +1/-1 array: alone (reads 4 B per element)
    # and fused into the stored inclusive scan
    res = torch.empty(2, dtype=torch.int32, device="cuda")
    med, _ = time_events(lambda: ds.bracket_scan(d_in, result=res, store=False), reps, 3)
    out["bracket_check_2^28"] = row(n, med, 4 * n)
    med, _ = time_events(lambda: ds.bracket_scan(d_in, out=d_out, result=res), reps, 3)
    out["bracket_scan_2^28"] = row(n, med, 8 * n)
    # the same array negated: 98% of its running sums are negative, so most
    # warps find a negative value (the flag store must not queue up)
    d_in.neg_()
    med, _ = time_events(lambda: ds.bracket_scan(d_in, out=d_out, result=res), reps, 3)
    out["bracket_scan_2^28_mostly_negative"] = row(n, med, 8 * n)
    d_in.neg_()
    # the fold alone (one read, 4 B per element), and one rank's device work
    # in the sharded scan (its total, the fold of the gathered totals, the
    # scan from the carry: 12 B per element); the exchange between ranks is
    # not part of this single-GPU row
    tot = torch.empty(1, dtype=torch.int32, device="cuda")
    med, _ = time_events(lambda: ds.reduce(d_in, out=tot), reps, 3)
    out["reduce_i32_add_2^28"] = row(n, med, 4 * n)
    med, _ = time_events(lambda: ds.sharded_scan(d_in, d_out), reps, 3)
    out["sharded_scan_one_rank_2^28"] = row(n, med, 12 * n)
    del d_in
    xm = torch.from_numpy(wl.max_values(n)).cuda()
    med, _ = time_events(lambda: ds.scan_inclusive(xm, d_out, op="max"), reps, 3)
    out["i32_max_inclusive_2^28"] = row(n, med, 8 * n)
    xm.copy_(torch.from_numpy(wl.xor_values(n).view(np.int32)))
    med, _ = time_events(lambda: ds.scan_inclusive(xm, d_out, op="xor", as_uint32=True), reps, 3)
    out["u32_xor_inclusive_2^28"] = row(n, med, 8 * n)
    ds.set_carry_mode("rts")
    med, _ = time_events(lambda: ds.scan_exclusive(xm, d_out), reps, 3)
    out["i32_add_exclusive_2^28_reduce_then_scan"] = row(n, med, 8 * n)
    ds.set_carry_mode(args.carry)
    del xm
    # segmented add at N = 2^28 (heads at rate 1/1024): 5 B read + 4 B written
    sv, sh = wl.segmented(n)
    dsv = torch.from_numpy(sv).cuda()
    dsh = torch.from_numpy(sh).cuda()
    del sv, sh
    med, _ = time_events(lambda: ds.segmented_scan_inclusive(dsv, dsh, d_out), reps, 3)
    out["segmented_i32_add_inclusive_2^28"] = row(n, med, 9 * n)
    med, _ = time_events(lambda: ds.segmented_scan_exclusive(dsv, dsh, d_out), reps, 3)
    out["segmented_i32_add_exclusive_2^28"] = row(n, med, 9 * n)
    del dsv, dsh, d_out

    # compaction at N = 2^26
    nc = wl.N_COMPACT
    v = wl.compaction_values(nc)
    dv = torch.from_numpy(v).cuda()
    dout = torch.empty_like(dv)
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    comp, comp_gt = {}, {}
    for sel in wl.SELECTIVITIES:
        f = torch.from_numpy(wl.predicate_flags(v, wl.threshold_for(sel))).cuda()
        med, _ = time_events(lambda: ds.compact(dv, f, dout, cnt), reps, 3)
        k = int(cnt.item())
        r = row(nc, med, 5 * nc + 4 * k + 4)
        r["kept"] = k
        comp[f"{int(sel * 100)}%"] = r
        del f
        t = wl.threshold_for(sel)
        med, _ = time_events(lambda: ds.compact_greater(dv, t, dout, cnt), reps, 3)
        k = int(cnt.item())
        r = row(nc, med, 4 * nc + 4 * k + 4)
        r["kept"] = k
        comp_gt[f"{int(sel * 100)}%"] = r
    out["compaction_2^26"] = comp
    out["compaction_gt_fused_2^26"] = comp_gt
    # the fused predicate's two-launch form (measurement hook)
    comp_gt2 = {}
    ds.set_carry_mode("l2")
    for sel in wl.SELECTIVITIES:
        t = wl.threshold_for(sel)
        med, _ = time_events(lambda: ds.compact_greater(dv, t, dout, cnt), reps, 3)
        k = int(cnt.item())
        r = row(nc, med, 4 * nc + 4 * k + 4)
        r["kept"] = k
        comp_gt2[f"{int(sel * 100)}%"] = r
    ds.set_carry_mode(args.carry)
    out["compaction_gt_fused_two_launch_2^26"] = comp_gt2
    # the pipelined form alone (the default tries the one-pass capture first)
    comp_gt3 = {}
    ds.set_carry_mode("pipelined")
    for sel in wl.SELECTIVITIES:
        t = wl.threshold_for(sel)
        med, _ = time_events(lambda: ds.compact_greater(dv, t, dout, cnt), reps, 3)
        k = int(cnt.item())
        r = row(nc, med, 4 * nc + 4 * k + 4)
        r["kept"] = k
        comp_gt3[f"{int(sel * 100)}%"] = r
    ds.set_carry_mode(args.carry)
    out["compaction_gt_fused_pipelined_2^26"] = comp_gt3

    # split and radix sort at N = 2^26
    keys = torch.from_numpy(wl.radix_keys(nc).view(np.int32)).cuda()
    med, _ = time_events(lambda: ds.split_bit(keys, 17, dout), reps, 3)
    out["split_bit_2^26"] = row(nc, med, 12 * nc)
    work = torch.empty_like(keys)
    tmp = torch.empty_like(keys)
    sreps = max(3, reps // 4)

    def sort_once():
        work.copy_(keys)
        ds.radix_sort(work, tmp)
    copy_med, _ = time_events(lambda: work.copy_(keys), sreps, 2)
    med, _ = time_events(sort_once, sreps, 2)
    sort_ms = med - copy_med
    out["radix_sort_32pass_2^26"] = {"ms": round(sort_ms, 3), "gelem_s": round(nc / (sort_ms / 1e3) / 1e9, 2),
                                     "gbs": round((32 * 8 * nc + 4 * nc) / (sort_ms / 1e3) / 1e9, 1),
                                     "frac": round((32 * 8 * nc + 4 * nc) / (sort_ms / 1e3) / 1e9 / peak, 4)}
    def sort_digits_once():
        work.copy_(keys)
        ds.radix_sort_digits(work, tmp)
    med, _ = time_events(sort_digits_once, sreps, 2)
    sort_ms = med - copy_med
    digit_bytes = 4 * 12 * nc   # 4 passes: count read, scatter read and write
    out["radix_sort_8bit_4pass_2^26"] = {"ms": round(sort_ms, 3), "gelem_s": round(nc / (sort_ms / 1e3) / 1e9, 2),
                                         "gbs": round(digit_bytes / (sort_ms / 1e3) / 1e9, 1),
                                         "frac": round(digit_bytes / (sort_ms / 1e3) / 1e9 / peak, 4)}
    del dv, dout, keys, work, tmp

    # fp32 add at N = 2^24 (128 MB of traffic: L2 flushed between reps)
    xf = torch.from_numpy(wl.unit_floats()).cuda()
    yf = torch.empty_like(xf)
    nf = xf.numel()
    # per-call events snap to the timer's ~2 us ticks: many calls, trimmed mean
    flushed_reps = max(reps, 200)
    _, mean = time_events(lambda: ds.scan_inclusive(xf, yf), flushed_reps, 3, flush=flush)
    out["f32_add_inclusive_2^24"] = row(nf, mean, 8 * nf)
    _, mean = time_events(lambda: ds.scan_exclusive(xf, yf), flushed_reps, 3, flush=flush)
    out["f32_add_exclusive_2^24"] = row(nf, mean, 8 * nf)
    del xf, yf

    # N = 65,536 latency (launch-bound)
    xs = torch.from_numpy(wl.small_digits()).cuda()
    ys = torch.empty_like(xs)
    _, mean = time_events(lambda: ds.scan_exclusive(xs, ys), flushed_reps, 3, flush=flush)
    out["i32_add_exclusive_65536"] = row(xs.numel(), mean, 8 * xs.numel())
    return out


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from stream_compaction_device_gb300 import workloads as wl
    n = args.n
    x = wl.brackets(n)
    # each step scans the whole array (about 0.22 s at 2^28 on one core)
    # unless steps + warm-up would run past REF_FULL_STEPS full scans; then
    # every step scans the same leading sample, sized to that budget
    calls = args.steps + args.warmup
    m = n if calls <= REF_FULL_STEPS else max(4096, (n * REF_FULL_STEPS // calls) // 4096 * 4096)
    xs = x[:m]
    for _ in range(args.warmup):
        oracle.scan(xs, "add", False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan(xs, "add", False)
    el = time.perf_counter() - t0
    value = m * args.steps / el / 1e9
    if m == n:
        sample = (f"serial oracle exclusive add-scan of the whole 2^{n.bit_length() - 1}-element workload per step, "
                  f"{args.steps} steps, one thread")
    else:
        sample = (f"serial oracle exclusive add-scan of the workload's first {m} elements per step "
                  f"({args.steps} steps + {args.warmup} warm-up would exceed {REF_FULL_STEPS} whole scans), "
                  "one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "Gelem/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": {"workload": f"int32 exclusive add-scan, N=2^{n.bit_length() - 1}, +1/-1 bracket sequence "
                               "(p=0.5, seed 3)", "n": n, "op": "add", "inclusive": False},
        "cpu_baseline": {"value": round(value, 4), "unit": "Gelem/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_op(args):
    """One library call at ``--n`` elements, ``--warmup`` + ``--steps`` times
    back to back, for profiling a single kernel (``ncu -k ... -s W -c 1``):
    prints the per-call time, which is not a bench line."""
    import torch
    import stream_compaction_device_gb300 as ds
    from stream_compaction_device_gb300 import workloads as wl
    ds.load()
    if args.carry != "default":
        ds.set_carry_mode(args.carry)
    n = args.n
    if args.op == "compact50":
        v = wl.compaction_values(n)
        dv = torch.from_numpy(v).cuda()
        f = torch.from_numpy(wl.predicate_flags(v, wl.threshold_for(0.5))).cuda()
        out, cnt = torch.empty_like(dv), torch.empty(1, dtype=torch.int32, device="cuda")
        fn = lambda: ds.compact(dv, f, out, cnt)
    elif args.op in ("compact_gt1", "compact_gt50"):
        dv = torch.from_numpy(wl.compaction_values(n)).cuda()
        t = wl.threshold_for(0.01 if args.op == "compact_gt1" else 0.5)
        out, cnt = torch.empty_like(dv), torch.empty(1, dtype=torch.int32, device="cuda")
        fn = lambda: ds.compact_greater(dv, t, out, cnt)
    elif args.op == "f32scan":
        x = torch.from_numpy(wl.unit_floats(n)).cuda()
        out = torch.empty_like(x)
        fn = lambda: ds.scan_inclusive(x, out)
    elif args.op == "segscan":
        sv, sh = wl.segmented(n)
        dv, dh = torch.from_numpy(sv).cuda(), torch.from_numpy(sh).cuda()
        out = torch.empty_like(dv)
        fn = lambda: ds.segmented_scan_inclusive(dv, dh, out)
    elif args.op == "bracket_check":
        x = torch.from_numpy(wl.brackets(n)).cuda()
        res = torch.empty(2, dtype=torch.int32, device="cuda")
        fn = lambda: ds.bracket_scan(x, result=res, store=False)
    elif args.op == "split":
        keys = torch.from_numpy(wl.radix_keys(n).view(np.int32)).cuda()
        out = torch.empty_like(keys)
        fn = lambda: ds.split_bit(keys, 17, out)
    elif args.op == "sort32":
        keys = torch.from_numpy(wl.radix_keys(n).view(np.int32)).cuda()
        work, tmp = torch.empty_like(keys), torch.empty_like(keys)
        def fn():
            work.copy_(keys)
            ds.radix_sort(work, tmp)
    else:   # digit_sort
        keys = torch.from_numpy(wl.radix_keys(n).view(np.int32)).cuda()
        work, tmp = torch.empty_like(keys), torch.empty_like(keys)
        def fn():
            work.copy_(keys)
            ds.radix_sort_digits(work, tmp)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    b.synchronize()
    print(json.dumps({"op": args.op, "n": n, "ms_per_call": round(a.elapsed_time(b) / max(args.steps, 1), 5),
                      "status": ds.device_status(), "note": "single-op run for profiling; not a bench line"}))


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default: 3000 for this library, 20 for the reference arm)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--n", type=int, default=N_HEADLINE)
    p.add_argument("--carry", choices=["default", "lookback", "rts", "pipelined"], default="default")
    p.add_argument("--extra-reps", type=int, default=20)
    p.add_argument("--cpu-budget", type=float, default=10.0)
    p.add_argument("--no-extras", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--op", choices=["scan", "f32scan", "compact50", "compact_gt1", "compact_gt50", "segscan",
                                    "bracket_check", "split", "sort32",
                                    "digit_sort"],
                   default="scan", help="scan: the benchmark; the others run one call repeatedly for profiling")
    args = p.parse_args(argv)
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 3000
    if args.warmup < 3 and args.impl == "ours":
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.op != "scan":
        run_op(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
