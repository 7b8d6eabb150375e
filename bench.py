#!/usr/bin/env python3
"""Benchmark of the librcc hot path on one GB300 (or N independent replicas).

Workload: 8 logical ranks x 2^24 fp32 elements per rank (64 MiB each),
gradient-like values N(0, 1e-2) with 0.1% of elements scaled x100, drawn on
the device from fixed seeds.  One step is one pass of the whole hot path over
that batch:
  all_reduce sum, all_reduce mean, all_reduce max   (deterministic rank order)
  reduce (sum) to root 7, broadcast from root 0
  reduce_scatter (sum, shard 2^21), all_gather of those shards
  grad_sync_adamw: the 8 rank buffers as the gradients of one 2^24-element
    parameter tensor -> mean, unscale, fan-in-1024 statistics, 12-byte report,
    clip, AdamW update (one fp32 state copy)
Metric (value): all_reduce algorithm GB/s = 3 * R*N*bytes / (time of the
step's three all_reduce rows), those rows launched K times back to back
between one CUDA-event pair.  The whole step (K steps of all eight rows, also
back to back) is reported beside it (ms_per_step, step_algbw_gbs), and so is
the grad-sync row alone, K calls back to back (grad_sync_row); a separate pass
with an event between rows gives the per-row breakdown (rows).
Every input (512 MiB per row) exceeds the 129 MB L2, so no flush is needed.

After the timed step the same line carries, each timed on its own:
  bf16_rs_ag_8x2p26  reduce_scatter then all_gather, 8 ranks x 2^26 bf16 per
                     rank (shard 2^23), fp32 accumulation
  grad_sync_1024     gradient sync + AdamW over 4 ranks and 1024 fp32 tensors
                     (sizes log-uniform in [1024, 4194304]), default flow, with
                     4 state copies (one per rank) and with 1

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch under torchrun: each rank runs the same workload on its own
GPU (replicas; no data-path collective); the timed region is bracketed by
barriers and the max over ranks is reported.
"""
import argparse
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

R = 8
N = 1 << 24
ES = 4
ALG_BYTES_ROW = R * N * ES                     # R * N * s, one collective row
ROWS = ["all_reduce_sum", "all_reduce_mean", "all_reduce_max", "reduce", "broadcast",
        "reduce_scatter", "all_gather", "grad_sync_adamw"]
# minimum HBM traffic of each row (bytes)
MIN_TRAFFIC = {
    "all_reduce_sum": 2 * R * N * ES, "all_reduce_mean": 2 * R * N * ES,
    "all_reduce_max": 2 * R * N * ES,
    "reduce": (R + 1) * N * ES, "broadcast": (1 + R) * N * ES,
    "reduce_scatter": R * N * ES + N * ES, "all_gather": N * ES + R * N * ES,
    # stats pass: R reads + mean-grad write; update: mean-grad read + p, m, v read+write
    "grad_sync_adamw": (R * ES + ES) * N + (ES + 24) * N,
}
METRIC = "all_reduce algorithm GB/s and % of GB300 HBM roofline vs R, N, dtype (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0        # HBM3e data-sheet figure, for context only
WORKLOAD = "8 ranks x 2^24 fp32 per rank, gradient-like N(0,1e-2) + 0.1% x100"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="leave out the bf16 RS/AG and 1024-tensor grad-sync legs of the line")
    ap.add_argument("--case", default="step",
                    choices=["step", "all_reduce", "reduce", "broadcast", "reduce_scatter",
                             "all_gather", "all_to_all", "grad_sync", "grad_sync_1024",
                             "all_reduce_rank", "checkpoint"],
                    help="step: the whole hot path (the benchmark line); otherwise time one "
                         "collective alone on --ranks x --elems (profiling and sweeps)")
    ap.add_argument("--ranks", type=int, default=R)
    ap.add_argument("--elems", type=int, default=N)
    ap.add_argument("--dtype", default="f32", choices=["f32", "bf16"])
    ap.add_argument("--op", default="sum", choices=["sum", "mean", "max", "min"])
    ap.add_argument("--fast", action="store_true", help="pairwise-tree sums instead of rank order")
    ap.add_argument("--replicas", type=int, default=1, help="optimizer-state copies (grad_sync_1024)")
    ap.add_argument("--hier", type=int, default=None, choices=[0, 1],
                    help="grad-sync statistics: 1 fan-in-1024 combines, 0 flat "
                         "(default: the binding's default, 1)")
    ap.add_argument("--elems-per-row", type=int, default=0,
                    help="statistics row size for the grad-sync cases (0: the library default)")
    ap.add_argument("--sweep", action="store_true",
                    help="size sweep: all_reduce mean (fp32, bf16), broadcast root 0 and reduce "
                         "root R-1 for R in {2,4,8}, N = 257*4^k and 2^28; one JSON line per point")
    ap.add_argument("--gs-mode", default="host", choices=["host", "device", "graph", "multi", "host_graph"],
                    help="grad-sync decision: host readback (default), device kernel, or device "
                         "kernel + captured update launches")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def combine_ranks(local_ms, local_units, world, device="cpu"):
    """Max of the per-rank times and sum of the per-rank work over the group."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ environment facts

def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            v = d.get(key)
            if isinstance(v, dict):     # {"burst": ..., ...}: a kernel timed alone
                v = v.get("burst", v.get("value"))
            if isinstance(v, (int, float)) and v > 0:
                return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("collectives.cuh", "collectives_part.cu"):
        with open(os.path.join(ROOT, "gradient_sync_rcc_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """Per-launch DRAM bytes of the all_reduce kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "all_reduce_f32_8x2p24_ncu.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"kernel-source-sha256-16:\s*([0-9a-f]+)", text)
    tb = re.search(r"traffic-bytes-per-launch:\s*([0-9]+)", text)
    if not sha or not tb or sha.group(1) != kernel_source_sha():
        return None
    return int(tb.group(1))


class ClockSampler:
    # One query field holds every throttle reason: the reasons bitmask, whose
    # bits are NVML's clocks-event reasons.
    FIELDS = "clocks.sm,clocks.max.sm,clocks_event_reasons.active"
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def close(self):
        """Ends the child if it still runs (stop() has not been reached)."""
        if self.proc is not None and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def lines(self):
        """Sample lines written so far (the file is shared with the child)."""
        if self.f is None:
            return 0
        self.f.flush()
        with open("/proc/self/fd/%d" % self.f.fileno()) as g:
            return sum(1 for _ in g)

    def stop(self, first_line=0):
        """Summarise the samples from line `first_line` on (the timed region);
        if that window holds none, the load pre-roll's samples stand in."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.seek(0)
        all_lines = self.f.read().splitlines()
        window = "timed region"
        chosen = all_lines[first_line:]
        if not any(len(l.split(",")) >= 3 for l in chosen):
            chosen, window = all_lines, "load pre-roll and timed region"
        sm, mx, reasons = [], [], set()
        for line in chosen:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 3:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                mask = int(parts[2], 16)
            except ValueError:
                continue
            for bit, name in self.REASON_BITS.items():
                if mask & bit:
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "window": window,
                "interval_ms": 100}


# ------------------------------------------------------------------ our arm

class Workload:
    def __init__(self, device):
        import torch
        from gradient_sync_rcc_gb300 import rcc, synth
        self.torch, self.rcc = torch, rcc
        self.dev = device
        self.ins = synth.gpu_rank_buffers("grad", R, N, torch.float32, (2, 1), device)
        self.ar = [torch.empty(N, device=device) for _ in range(R)]
        self.red = torch.empty(N, device=device)
        self.bc = [torch.empty(N, device=device) for _ in range(R)]
        self.rs = [torch.empty(N // R, device=device) for _ in range(R)]
        self.ag = [torch.empty(N, device=device) for _ in range(R)]
        p0 = synth.gpu_draw("normal:0.02", N, torch.float32, (2, 2), device)
        self.gs_tensors = [dict(grads=self.ins, params=[p0], exp_avg=[torch.zeros(N, device=device)],
                                exp_avg_sq=[torch.zeros(N, device=device)],
                                mean_grad=torch.empty(N, device=device))]
        self.sets = rcc.ParamSets(self.gs_tensors)
        self.cfg = rcc.adamw_cfg(replicas=1, max_grad_norm=1.0)
        self.state = rcc.optim_state(scale=1.0)

    def step(self, h, events=None, ins=None, sets=None):
        """One pass of every row over the rank buffers `ins` (default: the
        resident workload); `sets` is the matching gradient ParamSets."""
        rcc = self.rcc
        ins = self.ins if ins is None else ins
        sets = self.sets if sets is None else sets

        def mark(i):
            if events is not None:
                events[i].record()

        mark(0)
        rcc.all_reduce(h, ins, self.ar, "sum")
        mark(1)
        rcc.all_reduce(h, ins, self.ar, "mean")
        mark(2)
        rcc.all_reduce(h, ins, self.ar, "max")
        mark(3)
        rcc.reduce(h, ins, self.red, root=R - 1, op="sum")
        mark(4)
        rcc.broadcast(h, ins[0], self.bc, root=0)
        mark(5)
        rcc.reduce_scatter(h, ins, self.rs, "sum")
        mark(6)
        rcc.all_gather(h, self.rs, self.ag)
        mark(7)
        rep = rcc.grad_sync_adamw(h, sets, self.cfg, self.state)
        mark(8)
        return rep

    def grad_sync_row(self, h):
        """The step's grad-sync row alone."""
        return self.rcc.grad_sync_adamw(h, self.sets, self.cfg, self.state)

    def ar_rows(self, h):
        """The metric's rows alone: the step's three all_reduce rows."""
        rcc = self.rcc
        rcc.all_reduce(h, self.ins, self.ar, "sum")
        rcc.all_reduce(h, self.ins, self.ar, "mean")
        rcc.all_reduce(h, self.ins, self.ar, "max")


def e2e_leg(torch, rcc, wl, h, K, ar_only=False):
    """End to end through the public API with host buffers: every step copies
    its R input buffers from pinned host memory and reads a result back
    (rank 0's all_reduce output and, in the whole step, inside the grad-sync
    call, the 12-byte report).  ar_only: the step is the three all_reduce rows
    (the metric's rows); otherwise all eight rows.  Inputs are double-buffered:
    step k+1's copies run on four copy streams while step k computes.  Returns
    ms per step."""
    sets_in = [wl.ins, [torch.empty_like(x) for x in wl.ins]]
    gs_sets = [wl.sets, rcc.ParamSets([dict(wl.gs_tensors[0], grads=sets_in[1])])]
    host_in = [torch.empty(N, dtype=torch.float32, pin_memory=True) for _ in range(R)]
    for x, d in zip(host_in, wl.ins):
        x.copy_(d)
    host_out = torch.empty(N, dtype=torch.float32, pin_memory=True)
    main = torch.cuda.current_stream()
    nstreams = 4
    copy_streams = [torch.cuda.Stream() for _ in range(nstreams)]
    copied = [[torch.cuda.Event() for _ in range(nstreams)] for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def issue_copy(k):
        b = k % 2
        for j, cs in enumerate(copy_streams):
            if used[b]:
                cs.wait_event(consumed[b])   # the step that last read buffer set b is done
            with torch.cuda.stream(cs):
                for i in range(j, R, nstreams):
                    sets_in[b][i].copy_(host_in[i], non_blocking=True)
            copied[b][j].record(cs)

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    issue_copy(0)
    for k in range(K):
        b = k % 2
        if k + 1 < K:
            issue_copy(k + 1)
        for ev in copied[b]:
            main.wait_event(ev)
        if ar_only:
            for op in ("sum", "mean", "max"):
                rcc.all_reduce(h, sets_in[b], wl.ar, op)
        else:
            wl.step(h, ins=sets_in[b], sets=gs_sets[b])
        consumed[b].record(main)
        used[b] = True
        host_out.copy_(wl.ar[0], non_blocking=True)
    torch.cuda.synchronize()
    return (time.perf_counter() - t0) * 1e3 / K


def copy_bandwidth(torch, device):
    """D2D copy of 2 GiB (read + write counted), for context only."""
    a = torch.empty(1 << 29, dtype=torch.float32, device=device)
    b = torch.empty_like(a)
    for _ in range(3):
        b.copy_(a)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(10):
        b.copy_(a)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / 10
    del a, b
    return 2 * (1 << 31) / (ms * 1e-3) / 1e9


def timed_batch(torch, fn, K, warm=3):
    """Mean ms of K back-to-back calls of fn on the current stream, between one
    pair of CUDA events.  An event recorded between two launches costs the
    device about 2 us and breaks programmatic dependent launch (another ~2 us
    of launch latency no longer hidden), so the collectives are timed this way;
    the per-call median below keeps an event between calls."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / K


def timed_median(torch, fn, K, warm=3):
    """Median of K CUDA-event-timed calls of fn on the current stream."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    ev[0].record()
    for k in range(K):
        fn()
        ev[k + 1].record()
    torch.cuda.synchronize()
    return statistics.median(ev[k].elapsed_time(ev[k + 1]) for k in range(K))


def _row(ms, alg_bytes, traffic, peak, src):
    gbs = traffic / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "algbw_gbs": round(alg_bytes / (ms * 1e-3) / 1e9, 1),
            "min_traffic_bytes": traffic, "traffic_gbs": round(gbs, 1),
            "frac_of_" + src: round(gbs / peak, 4)}


def bf16_rs_ag_leg(torch, rcc, dev_index, device, peak, src, K=10):
    """reduce_scatter then all_gather, 8 ranks x 2^26 bf16 per rank, N(0, 1)
    inputs, fp32 accumulation, rank-order sums; each collective timed alone
    (K launches back to back).  Minimum traffic (R + 1) * N * 2 bytes for both."""
    from gradient_sync_rcc_gb300 import synth
    R3, N3 = 8, 1 << 26
    n3 = N3 // R3
    ins = synth.gpu_rank_buffers("normal1", R3, N3, torch.bfloat16, (300,), device)
    rs = [torch.empty(n3, dtype=torch.bfloat16, device=device) for _ in range(R3)]
    ag = [torch.empty(N3, dtype=torch.bfloat16, device=device) for _ in range(R3)]
    h = rcc.register(dev_index, R3, rcc.BF16, True)
    try:
        rs_ms = timed_batch(torch, lambda: rcc.reduce_scatter(h, ins, rs, "sum"), K)
        ag_ms = timed_batch(torch, lambda: rcc.all_gather(h, rs, ag), K)
    finally:
        rcc.finish(h)
    traffic = (R3 + 1) * N3 * 2
    return {"workload": "8 ranks x 2^26 bf16 per rank (shard 2^23), N(0,1), fp32 accumulation, "
                        "rank order; %d back-to-back launches each between one event pair" % K,
            "reduce_scatter": _row(rs_ms, R3 * N3 * 2, traffic, peak, src),
            "all_gather": _row(ag_ms, R3 * N3 * 2, traffic, peak, src)}


def grad_sync_1024_leg(torch, rcc, dev_index, device, peak, src, K=5, replicas=(4, 1)):
    """Gradient sync + AdamW: 4 ranks, 1024 fp32 tensors with sizes
    log-uniform in [1024, 4194304] (429,088,269 elements), grads
    N(0, 1e-3) x 65536, lr 1e-3, betas (0.9, 0.999), eps 1e-8, wd 0.01,
    max_grad_norm 1.0, the mean gradient stored; default flow (report read
    back, decision on the host, one update launch per tensor).  Per state-copy
    count: 3 untimed steps, then the median of K CUDA-event-timed steps.
    Minimum traffic per element (4R + 4) + (4 + 24 * replicas) bytes."""
    from gradient_sync_rcc_gb300 import synth
    Rk, P = 4, 1024
    sizes = synth.param_sizes(P, 1024, 4194304, 20)
    E = sum(sizes)
    grads = [[synth.gpu_draw("normal:1e-3", n, torch.float32, (22, i, 1, r), device) * 65536.0
              for r in range(Rk)] for i, n in enumerate(sizes)]
    means = [torch.empty(n, device=device) for n in sizes]
    out = {"workload": "4 ranks, 1024 fp32 tensors log-uniform in [1024, 4194304], %d elements, "
                       "default flow, median of %d steps after 3" % (E, K)}
    for rep in replicas:
        tensors = []
        for i, n in enumerate(sizes):
            p0 = synth.gpu_draw("normal:0.02", n, torch.float32, (21, i), device)
            tensors.append(dict(grads=grads[i], params=[p0] + [p0.clone() for _ in range(rep - 1)],
                                exp_avg=[torch.zeros(n, device=device) for _ in range(rep)],
                                exp_avg_sq=[torch.zeros(n, device=device) for _ in range(rep)],
                                mean_grad=means[i]))
        sets = rcc.ParamSets(tensors)
        cfg = rcc.adamw_cfg(replicas=rep)
        state = rcc.optim_state(scale=65536.0)
        h = rcc.register(dev_index, Rk, rcc.F32, True)
        try:
            ms = timed_median(torch, lambda: rcc.grad_sync_adamw(h, sets, cfg, state), K)
        finally:
            rcc.finish(h)
        traffic = (Rk * 4 + 4) * E + (4 + 24 * rep) * E
        row = _row(ms, Rk * E * 4, traffic, peak, src)
        row.pop("algbw_gbs")
        out["replicas_%d" % rep] = row
        del tensors, sets
        torch.cuda.empty_cache()
    return out


def bench_ours(args):
    import torch
    from gradient_sync_rcc_gb300 import build, rcc
    rank, world, local = dist_env()
    build.build()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    device = "cuda:%d" % local
    # The clock sampler starts first and the load pre-roll below runs until it
    # has been up 1.5 s: on a fresh box the first nvidia-smi instance stalled
    # a saturated GPU for 60-140 ms about a second after it started.
    sampler = ClockSampler(local)
    sampler.start()
    t_sampler = time.perf_counter()
    h = None
    try:
        wl = Workload(device)
        h = rcc.register(local, R, rcc.F32, True)
        for _ in range(max(args.warmup, 3)):
            wl.step(h)
        torch.cuda.synchronize()
        K = args.steps
        Kr = min(K, 20)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ROWS) + 1)]
              for _ in range(Kr)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ar_start = torch.cuda.Event(enable_timing=True)
        ar_end = torch.cuda.Event(enable_timing=True)
        gs_start = torch.cuda.Event(enable_timing=True)
        gs_end = torch.cuda.Event(enable_timing=True)
        # load pre-roll: keep stepping (untimed) until the clock sampler is up
        # and has run 1.5 s
        t_pre = time.perf_counter()
        while sampler.proc is not None and time.perf_counter() - t_pre < 5.0:
            for _ in range(20):
                wl.step(h)
            torch.cuda.synchronize()
            if sampler.lines() >= 2 and time.perf_counter() - t_sampler >= 1.5:
                break
        first_line = sampler.lines()
        # timed region 1: K steps, every row launched back to back
        launches0 = rcc.launch_count()
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        for k in range(K):
            wl.step(h)
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        # timed region 2: the metric's three all_reduce rows, K times back to back
        launches1 = rcc.launch_count()
        barrier(world)
        torch.cuda.synchronize()
        ar_start.record()
        for k in range(K):
            wl.ar_rows(h)
        ar_end.record()
        torch.cuda.synchronize()
        barrier(world)
        launches2 = rcc.launch_count()
        # timed region 3: the grad-sync row, K calls back to back
        barrier(world)
        torch.cuda.synchronize()
        gs_start.record()
        for k in range(K):
            wl.grad_sync_row(h)
        gs_end.record()
        torch.cuda.synchronize()
        barrier(world)
        launches3 = rcc.launch_count()
        clocks = sampler.stop(first_line)
        ms_total = start.elapsed_time(end)
        ar_ms_sum = ar_start.elapsed_time(ar_end) / K      # the three rows, per iteration
        gs_ms = gs_start.elapsed_time(gs_end) / K
        # per-row breakdown (not a headline figure): Kr more steps with an event
        # between rows, which adds about 2-4 us of device time to each row
        for k in range(Kr):
            wl.step(h, ev[k])
        torch.cuda.synchronize()
        row_ms = {name: statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(Kr))
                  for i, name in enumerate(ROWS)}

        # end to end: inputs from pinned host memory, result read back, every step
        Ke = max(3, min(K, 50))
        barrier(world)
        e2e_ar_ms = e2e_leg(torch, rcc, wl, h, Ke, ar_only=True)
        barrier(world)
        e2e_ms = e2e_leg(torch, rcc, wl, h, Ke)
        barrier(world)
    finally:
        sampler.close()
        if h is not None:
            rcc.finish(h)
    peak0, src0 = peak_hbm()
    del wl
    torch.cuda.empty_cache()
    extra = {}
    if not args.no_extra:
        extra["bf16_rs_ag_8x2p26"] = bf16_rs_ag_leg(torch, rcc, local, device, peak0, src0)
        torch.cuda.empty_cache()
        extra["grad_sync_1024"] = grad_sync_1024_leg(torch, rcc, local, device, peak0, src0)
        torch.cuda.empty_cache()
    copy_gbs = copy_bandwidth(torch, device)

    ms_step = ms_total / K
    alg_step = ALG_BYTES_ROW * len(ROWS)
    ar_rows = ["all_reduce_sum", "all_reduce_mean", "all_reduce_max"]
    max_ar, total_ar = combine_ranks(ar_ms_sum, ALG_BYTES_ROW * len(ar_rows), world, device)
    max_step, total_step = combine_ranks(ms_step, alg_step, world, device)
    max_e2e, total_e2e = combine_ranks(e2e_ar_ms, ALG_BYTES_ROW * len(ar_rows), world, device)
    max_e2e_step, total_e2e_step = combine_ranks(e2e_ms, alg_step, world, device)
    max_gs, _ = combine_ranks(gs_ms, 0, world, device)
    if rank != 0:
        return
    peak, peak_src = peak_hbm()
    ar_ms = ar_ms_sum / len(ar_rows)
    ar_traffic = MIN_TRAFFIC["all_reduce_sum"]
    achieved = ar_traffic / (ar_ms * 1e-3) / 1e9
    traffic = ncu_traffic()
    rows = {}
    for name in ROWS:
        t = row_ms[name]
        gbs = MIN_TRAFFIC[name] / (t * 1e-3) / 1e9
        rows[name] = {"ms": round(t, 4), "algbw_gbs": round(ALG_BYTES_ROW / (t * 1e-3) / 1e9, 1),
                      "traffic_gbs": round(gbs, 1), "frac_of_" + peak_src: round(gbs / peak, 4)}
    out = {
        "metric": METRIC,
        "value": round(total_ar / (max_ar * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(max_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded device draws)",
        "config": {"workload": WORKLOAD, "ranks": R, "elements_per_rank": N,
                   "rows_per_step": ROWS, "value_rows": ar_rows,
                   "mode": "deterministic rank order",
                   "adamw_replicas": 1, "l2": "inputs 512 MiB per row > 129 MB L2, no flush",
                   "timing": ("value: K iterations of the three all_reduce rows launched back "
                              "to back between one CUDA-event pair; ms_per_step: K steps of "
                              "all eight rows likewise; grad_sync_row: K grad-sync calls "
                              "likewise; rows: a separate pass of min(K, 20) steps with an "
                              "event between rows (each row about 2-4 us more)"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "step_algbw_gbs": round(total_step / (max_step * 1e-3) / 1e9, 2),
        "roofline": {"kernel": "all_reduce (multi-pointer pass, fp32, R=8, N=2^24)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "nominal_peak": NOMINAL_HBM_GBS, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "traffic_source": ("copied from the committed ncu summary "
                                        "profiles/all_reduce_f32_8x2p24_ncu.md, taken on the "
                                        "same kernel source" if traffic is not None else
                                        "null: no ncu summary taken on this kernel source"),
                     "algorithmic_bytes_per_launch": ar_traffic,
                     "avg_launch_ms": round(ar_ms, 4)},
        "rows": rows,
        "grad_sync_row": {"ms": round(max_gs, 4),
                          "traffic_gbs": round(MIN_TRAFFIC["grad_sync_adamw"] / (max_gs * 1e-3) / 1e9, 1),
                          "frac_of_" + peak_src: round(MIN_TRAFFIC["grad_sync_adamw"] / (max_gs * 1e-3)
                                                       / 1e9 / peak, 4),
                          "min_traffic_bytes": MIN_TRAFFIC["grad_sync_adamw"],
                          "timing": "the step's grad-sync row alone, K calls back to back "
                                    "between one event pair (each call reads its report back)"},
        "e2e": {"value": round(total_e2e / (max_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(max_e2e, 3),
                "what": "per step: the 8 rank inputs copied from pinned host memory, the "
                        "step's three all_reduce rows through the C ABI, one output read back",
                "pipeline": "inputs double-buffered; step k+1's H2D copies on 4 streams overlap step k",
                "h2d_bytes_per_step": R * N * ES, "d2h_bytes_per_step": N * ES},
        "e2e_step": {"value": round(total_e2e_step / (max_e2e_step * 1e-3) / 1e9, 2),
                     "unit": "GB/s (algorithm bytes of all eight rows)",
                     "ms_per_step": round(max_e2e_step, 3),
                     "what": "the whole step (all eight rows) with host inputs, as e2e",
                     "h2d_bytes_per_step": R * N * ES, "d2h_bytes_per_step": N * ES + 12},
        "gpu_launches": int(launches3 - launches0),
        "gpu_launches_per_region": {"step": int(launches1 - launches0),
                                    "value": int(launches2 - launches1),
                                    "grad_sync_row": int(launches3 - launches2)},
        "clocks": clocks,
        "d2d_copy_gbs_measured_here": round(copy_gbs, 1),
    }
    out.update(extra)
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(target_s=10.0)
        omp = cpu_baseline_omp(target_s=5.0)
        if omp is not None:
            out["cpu_baseline_omp"] = omp
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ the oracle on host cores

def oracle_step(orc, xs, state):
    """One pass of the step's rows over host arrays, in the oracle.  Returns
    the seconds spent in the three all_reduce rows (the metric's rows)."""
    n = xs[0].size
    t0 = time.perf_counter()
    for op in ("sum", "mean", "max"):
        orc.all_reduce(xs, op)
    t_ar = time.perf_counter() - t0
    out = np.empty(n, np.float32)
    orc.reduce(xs, "sum", out)
    orc.broadcast(xs[0], [np.empty(n, np.float32) for _ in range(len(xs))])
    rs = orc.reduce_scatter(xs, "sum")
    orc.all_gather(rs)
    p, m, v, sc, t = state
    t, _, _ = orc.grad_sync_adamw_step([xs], [p], [m], [v], lr=1e-3, beta1=0.9, beta2=0.999,
                                       eps=1e-8, weight_decay=0.01, max_grad_norm=1.0, step=t,
                                       scaler=sc)
    state[4] = t
    return t_ar


def host_info():
    """Host cores and CPU model, recorded beside every oracle timing."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.startswith("Model name:"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model, "machine": platform.machine()}


def _oracle_setup(n):
    import oracle as orc
    from gradient_sync_rcc_gb300 import synth
    orc.build.build()
    xs = synth.rank_buffers("grad", R, n, 2, 3)
    p = synth.normal(n, 0.02, 2, 4)
    state = [p, np.zeros(n, np.float32), np.zeros(n, np.float32), orc.scaler_new(1.0), 0]
    return orc, xs, state


def cpu_baseline(target_s=10.0, n=1 << 22):
    """The oracle as it stands, single-threaded, on a bounded sample of the
    workload: the step's eight rows over 8 ranks x n fp32; value in the
    metric's terms (the three all_reduce rows), the whole step beside it."""
    orc, xs, state = _oracle_setup(n)
    reps, t_ar = 0, 0.0
    t0 = time.perf_counter()
    while True:
        t_ar += oracle_step(orc, xs, state)
        reps += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return {"value": round(3 * R * n * ES * reps / t_ar / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "host": host_info(),
            "step_algbw_gbs": round(R * n * ES * len(ROWS) * reps / el / 1e9, 4),
            "sample": "the step's 8 rows over 8 ranks x 2^%d fp32 (1/%d of the workload), "
                      "%d passes, %.1f s single-threaded; value over the three all_reduce rows"
                      % (int(math.log2(n)), N // n, reps, el)}


def cpu_baseline_omp(target_s=5.0, n=1 << 22):
    """A second CPU baseline: the oracle's fp32 rank-order all_reduce
    arithmetic written with an OpenMP loop over elements, on every host core
    (oracle/rcc_oracle_omp.cpp; not part of the oracle's reference path).
    None if it cannot be built here."""
    try:
        import oracle.omp as omp
        lib = omp.lib()
    except Exception:
        return None
    from gradient_sync_rcc_gb300 import synth
    xs = synth.rank_buffers("grad", R, n, 2, 3)
    outs = [np.empty(n, np.float32) for _ in range(R)]
    threads = os.cpu_count() or 1
    reps, t_ar = 0, 0.0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < target_s:
        for op in ("sum", "mean", "max"):
            t1 = time.perf_counter()
            omp.all_reduce(xs, outs, op, threads)
            t_ar += time.perf_counter() - t1
        reps += 1
    return {"value": round(3 * R * n * ES * reps / t_ar / 1e9, 4), "unit": "GB/s",
            "cores": threads, "kind": "oracle arithmetic, OpenMP over elements",
            "host": host_info(),
            "sample": "the three all_reduce rows over 8 ranks x 2^%d fp32, %d passes on %d "
                      "threads" % (int(math.log2(n)), reps, threads)}


def bench_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    # each step is a bounded sample: 2^20 elements per rank (1/16 of the
    # workload) up to 250 steps, halved for each doubling of the step count
    # beyond that, so the whole run stays near a minute of host time
    K = args.steps
    shift = 0
    while shift < 4 and K > 250 << shift:
        shift += 1
    n = (1 << 20) >> shift
    orc, xs, state = _oracle_setup(n)
    for _ in range(max(args.warmup, 3)):
        oracle_step(orc, xs, state)
    t_ar = 0.0
    t0 = time.perf_counter()
    for _ in range(K):
        t_ar += oracle_step(orc, xs, state)
    el = time.perf_counter() - t0
    ms = el * 1e3 / K
    value = 3 * R * n * ES * K / t_ar / 1e9
    step_value = R * n * ES * len(ROWS) / (ms * 1e-3) / 1e9
    sample = ("each step: the 8 rows over 8 ranks x 2^%d fp32 (1/%d of the workload), "
              "single-threaded; value over the three all_reduce rows" % (20 - shift, 16 << shift))
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": world, "steps": K, "warmup": max(args.warmup, 3),
           "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded host draws)",
           "config": {"workload": WORKLOAD, "ranks": R, "elements_per_rank": N,
                      "rows_per_step": ROWS, "value_rows": ["all_reduce_sum", "all_reduce_mean",
                                                            "all_reduce_max"],
                      "mode": "deterministic rank order"},
           "step_algbw_gbs": round(step_value, 4),
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                            "kind": "oracle", "host": host_info(), "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def hier_kw(args):
    return {} if args.hier is None else {"hierarchical_stats": args.hier}


def gs_flags(rcc, mode):
    """`--gs-mode` -> rcc_adamw_cfg.flags."""
    return {"host": 0, "device": rcc.ADAMW_DEVICE_DECISION, "graph": rcc.ADAMW_GRAPH,
            "multi": rcc.ADAMW_DEVICE_DECISION | rcc.ADAMW_MULTI_TENSOR,
            "host_graph": rcc.ADAMW_HOST_GRAPH}[mode]


def bench_grad_sync_1024(args):
    """The gradient-sync workload: 4 ranks, 1024 fp32 tensors with sizes
    log-uniform in [1024, 4194304], grads N(0, 1e-3) x 65536, one AdamW step
    per iteration (the mean gradient is stored; `--replicas` state copies)."""
    import torch
    from gradient_sync_rcc_gb300 import build, rcc, synth
    build.build()
    dev = "cuda:0"
    Rk, P, rep = 4, 1024, args.replicas
    sizes = synth.param_sizes(P, 1024, 4194304, 20)
    E = sum(sizes)
    tensors = []
    for i, n in enumerate(sizes):
        g = [synth.gpu_draw("normal:1e-3", n, torch.float32, (22, i, 1, r), dev) * 65536.0
             for r in range(Rk)]
        p0 = synth.gpu_draw("normal:0.02", n, torch.float32, (21, i), dev)
        tensors.append(dict(grads=g, params=[p0.clone() for _ in range(rep)],
                            exp_avg=[torch.zeros(n, device=dev) for _ in range(rep)],
                            exp_avg_sq=[torch.zeros(n, device=dev) for _ in range(rep)],
                            mean_grad=torch.empty(n, device=dev)))
    sets = rcc.ParamSets(tensors)
    cfg = rcc.adamw_cfg(replicas=rep, flags=gs_flags(rcc, args.gs_mode),
                        elems_per_row=args.elems_per_row, **hier_kw(args))
    state = rcc.optim_state(scale=65536.0)
    h = rcc.register(0, Rk, rcc.F32, True)
    try:
        for _ in range(max(args.warmup, 3)):
            rcc.grad_sync_adamw(h, sets, cfg, state)
        torch.cuda.synchronize()
        K = args.steps
        l0 = rcc.launch_count()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        s.record()
        for _ in range(K):
            rep_ = rcc.grad_sync_adamw(h, sets, cfg, state)
        e.record()
        torch.cuda.synchronize()
        wall = (time.perf_counter() - t0) * 1e3 / K
        ms = s.elapsed_time(e) / K
        launches = (rcc.launch_count() - l0) // K
    finally:
        rcc.finish(h)
    traffic = (Rk * 4 + 4) * E + (4 + 24 * rep) * E
    peak, src = peak_hbm()
    out = {"case": "grad_sync_1024", "mode": args.gs_mode, "ranks": Rk, "tensors": P,
           "elements": E, "replicas": rep, "ms_per_step": round(ms, 3),
           "wall_ms_per_step": round(wall, 3),
           "launches_per_step": launches, "combine_launches": rep_.combine_launches,
           "min_traffic_bytes": traffic,
           "traffic_gbs": round(traffic / (ms * 1e-3) / 1e9, 1),
           "frac_of_" + src: round(traffic / (ms * 1e-3) / 1e9 / peak, 4)}
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = oracle_grad_sync_sample(tensors, sizes, Rk, rep, E)
    print(json.dumps(out), flush=True)


def oracle_grad_sync_sample(tensors, sizes, Rk, rep, E):
    """The oracle's step on this workload, streamed per tensor on host copies of
    a sample of the tensors (the first ones, at least 2^25 elements), scaled to
    the whole step by element count."""
    import oracle as orc
    orc.build.build()
    n_s, host = 0, []
    for i, n in enumerate(sizes):
        host.append(([t.cpu().numpy() for t in tensors[i]["grads"]],
                     tensors[i]["params"][0].cpu().numpy().copy(),
                     np.zeros(n, np.float32), np.zeros(n, np.float32)))
        n_s += n
        if n_s >= 1 << 25:
            break
    inv = np.float32(1.0 / 65536.0)
    t0 = time.perf_counter()
    st = orc.stats_new()
    means = []
    for g, _, _, _ in host:
        mean = orc.mean_unscale(g, inv)
        orc.stats_accumulate(st, mean)
        means.append(mean)
    d = orc.decide(st, 1.0)
    s = orc.adamw_scalars(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
    for _ in range(rep):
        for (_, p, m, v), mean in zip(host, means):
            orc.adamw_update(mean, d.clip_coef, s, p, m, v)
    el = time.perf_counter() - t0
    step_s = el * E / n_s
    traffic = (Rk * 4 + 4) * E + (4 + 24 * rep) * E
    return {"value_ms_per_step": round(step_s * 1e3, 1),
            "traffic_gbs": round(traffic / step_s / 1e9, 4), "cores": 1, "kind": "oracle",
            "host": host_info(),
            "sample": "first %d tensors (%d elements, %.2f s single-threaded), scaled by "
                      "element count to the %d-element step" % (len(host), n_s, el, E)}


def bench_case(args):
    """One collective alone, timed with CUDA events; prints one JSON line.  A
    collective's `ms` is the mean of K launches back to back (as in a stream
    of collectives); `median_ms` keeps an event between launches, which adds
    about 4 us to each."""
    import torch
    from gradient_sync_rcc_gb300 import build, rcc, synth
    build.build()
    dev = "cuda:0"
    Rk, n = args.ranks, args.elems
    dt = rcc.F32 if args.dtype == "f32" else rcc.BF16
    td = torch.float32 if dt == rcc.F32 else torch.bfloat16
    es = 4 if dt == rcc.F32 else 2
    c = args.case
    n_in = n // Rk if c == "all_gather" else n
    ins = synth.gpu_rank_buffers("uniform", Rk, n_in, td, (3, Rk, n), dev)
    if c == "reduce_scatter":
        outs = [torch.empty(n // Rk, dtype=td, device=dev) for _ in range(Rk)]
    elif c == "reduce":
        outs = torch.empty(n, dtype=td, device=dev)
    else:
        outs = [torch.empty(n, dtype=td, device=dev) for _ in range(Rk)]
    traffic = {"all_reduce": 2 * Rk * n * es, "reduce": (Rk + 1) * n * es,
               "broadcast": (Rk + 1) * n * es, "reduce_scatter": (Rk * n + n) * es,
               "all_gather": (n + Rk * n) * es, "all_to_all": 2 * Rk * n * es}.get(c)
    h = rcc.register(0, Rk, dt, not args.fast)
    sets = None
    if c == "grad_sync":
        p0 = synth.gpu_draw("normal:0.02", n, torch.float32, (3, 9), dev)
        sets = rcc.ParamSets([dict(grads=ins, params=[p0], exp_avg=[torch.zeros_like(p0)],
                                   exp_avg_sq=[torch.zeros_like(p0)],
                                   mean_grad=torch.empty_like(p0))])
        cfg = rcc.adamw_cfg(replicas=1, flags=gs_flags(rcc, args.gs_mode),
                            elems_per_row=args.elems_per_row, **hier_kw(args))
        state = rcc.optim_state(scale=1.0)
        traffic = (Rk * 4 + 4) * n + 28 * n

    def once():
        if c == "all_reduce":
            rcc.all_reduce(h, ins, outs, args.op)
        elif c == "reduce":
            rcc.reduce(h, ins, outs, root=Rk - 1, op=args.op)
        elif c == "broadcast":
            rcc.broadcast(h, ins[0], outs, root=0)
        elif c == "reduce_scatter":
            rcc.reduce_scatter(h, ins, outs, args.op)
        elif c == "all_gather":
            rcc.all_gather(h, ins, outs)
        elif c == "all_to_all":
            rcc.all_to_all_single(h, ins, outs)
        else:
            rcc.grad_sync_adamw(h, sets, cfg, state)

    try:
        for _ in range(max(args.warmup, 3)):
            once()
        torch.cuda.synchronize()
        K = args.steps
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        ev[0].record()
        for k in range(K):
            once()
            ev[k + 1].record()
        torch.cuda.synchronize()
        ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(K)]
        # a collective is timed as K launches back to back (timed_batch); the
        # grad-sync call, which waits on the host for its report, per call
        batch = timed_batch(torch, once, K, warm=0) if c != "grad_sync" else None
    finally:
        rcc.finish(h)
    peak, src = peak_hbm()
    med = statistics.median(ms)
    t = batch if batch is not None else med
    print(json.dumps({"case": c, "ranks": Rk, "elems": n, "dtype": args.dtype, "op": args.op,
                      "mode": "fast" if args.fast else "deterministic",
                      **({"gs_mode": args.gs_mode} if c == "grad_sync" else {}),
                      "ms": round(t, 5),
                      "timing": ("%d launches back to back between one event pair" % K
                                 if batch is not None else
                                 "median of %d calls, an event between calls" % K),
                      "median_ms": round(med, 5), "min_ms": round(min(ms), 5),
                      "algbw_gbs": round(Rk * n * es / (t * 1e-3) / 1e9, 1),
                      "traffic_gbs": round(traffic / (t * 1e-3) / 1e9, 1),
                      "frac_of_" + src: round(traffic / (t * 1e-3) / 1e9 / peak, 4),
                      "min_traffic_bytes": traffic}), flush=True)


def bench_rank_case(args):
    """all_reduce through the per-rank arrival API: one host thread and one
    CUDA stream per rank, each calling rcc_all_reduce_rank with its own
    buffers; the last rank to arrive launches the kernel, which waits for every
    rank's stream, and every rank's stream waits for it.  K rounds; the device
    time per round is taken on rank 0's stream between one event pair, the
    host time per round over all threads.  A second pass at 1,024 elements per
    rank gives the arrival protocol's own cost per round (host-bound)."""
    import threading
    import torch
    from gradient_sync_rcc_gb300 import build, rcc, synth
    build.build()
    dev = "cuda:0"
    Rk, K = args.ranks, args.steps
    peak, src = peak_hbm()

    def rounds(n, K):
        ins = synth.gpu_rank_buffers("uniform", Rk, n, torch.float32, (7, Rk, n), dev)
        outs = [torch.empty(n, device=dev) for _ in range(Rk)]
        streams = [torch.cuda.Stream() for _ in range(Rk)]
        h = rcc.register(0, Rk, rcc.F32, not args.fast)
        errs = []
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gate = threading.Barrier(Rk)

        def rank(r, nround, timed):
            try:
                s = streams[r]
                gate.wait()
                if timed and r == 0:
                    start.record(s)
                for _ in range(nround):
                    rcc.all_reduce_rank(h, r, ins[r], outs[r], args.op, stream=s)
                if timed and r == 0:
                    end.record(s)
            except BaseException as e:  # reported below
                errs.append(e)

        def run(nround, timed):
            ts = [threading.Thread(target=rank, args=(r, nround, timed)) for r in range(Rk)]
            t0 = time.perf_counter()
            for t in ts:
                t.start()
            for t in ts:
                t.join()
            torch.cuda.synchronize()
            return time.perf_counter() - t0

        try:
            torch.cuda.synchronize()
            run(3, False)                       # warm-up rounds
            wall = run(K, True)
        finally:
            rcc.finish(h)
        if errs:
            raise errs[0]
        return start.elapsed_time(end) / K, wall * 1e3 / K

    dev_ms, host_ms = rounds(args.elems, K)
    _, small_host_ms = rounds(1024, max(K, 200))
    traffic = 2 * Rk * args.elems * 4
    print(json.dumps({"case": "all_reduce_rank", "ranks": Rk, "elems": args.elems, "dtype": "f32",
                      "op": args.op, "mode": "fast" if args.fast else "deterministic",
                      "rounds": K, "ms": round(dev_ms, 5),
                      "timing": "rank 0's stream, K rounds between one event pair",
                      "host_ms_per_round": round(host_ms, 4),
                      "arrival_us_per_round_1024_elems": round(small_host_ms * 1e3, 1),
                      "algbw_gbs": round(Rk * args.elems * 4 / (dev_ms * 1e-3) / 1e9, 1),
                      "traffic_gbs": round(traffic / (dev_ms * 1e-3) / 1e9, 1),
                      "frac_of_" + src: round(traffic / (dev_ms * 1e-3) / 1e9 / peak, 4),
                      "min_traffic_bytes": traffic}), flush=True)


def bench_checkpoint(args):
    """Checkpoint save and restore of the 1,024-tensor optimizer state (4
    ranks, `--replicas` state copies) after one grad-sync step:
    checkpoint.state_dict copies params, exp_avg and exp_avg_sq to host
    arrays; load_state_dict copies them back into the device tensors.  Both
    are timed on the wall clock (each ends synchronised); the restored state
    is compared bit for bit with what was saved."""
    import torch
    from gradient_sync_rcc_gb300 import build, checkpoint, rcc, synth
    build.build()
    dev = "cuda:0"
    Rk, P, rep = 4, 1024, args.replicas
    sizes = synth.param_sizes(P, 1024, 4194304, 20)
    E = sum(sizes)
    tensors = []
    for i, n in enumerate(sizes):
        g = [synth.gpu_draw("normal:1e-3", n, torch.float32, (22, i, 1, r), dev) * 65536.0
             for r in range(Rk)]
        p0 = synth.gpu_draw("normal:0.02", n, torch.float32, (21, i), dev)
        tensors.append(dict(grads=g, params=[p0.clone() for _ in range(rep)],
                            exp_avg=[torch.zeros(n, device=dev) for _ in range(rep)],
                            exp_avg_sq=[torch.zeros(n, device=dev) for _ in range(rep)],
                            mean_grad=torch.empty(n, device=dev)))
    sets = rcc.ParamSets(tensors)
    cfg = rcc.adamw_cfg(replicas=rep)
    state = rcc.optim_state(scale=65536.0)
    h = rcc.register(0, Rk, rcc.F32, True)
    try:
        rcc.grad_sync_adamw(h, sets, cfg, state)
        torch.cuda.synchronize()
    finally:
        rcc.finish(h)
    nbytes = 3 * 4 * E * rep
    t0 = time.perf_counter()
    sd = checkpoint.state_dict(tensors, cfg, state)
    save_s = time.perf_counter() - t0
    for t in tensors:
        for k in ("params", "exp_avg", "exp_avg_sq"):
            for x in t[k]:
                x.zero_()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    checkpoint.load_state_dict(sd, tensors, rcc)
    torch.cuda.synchronize()
    load_s = time.perf_counter() - t0
    same = all(np.array_equal(x.cpu().numpy(), sd["tensors"][i][k][j])
               for i, t in enumerate(tensors) for k in ("params", "exp_avg", "exp_avg_sq")
               for j, x in enumerate(t[k]))
    print(json.dumps({"case": "checkpoint", "ranks": Rk, "tensors": P, "elements": E,
                      "replicas": rep, "state_bytes": nbytes,
                      "save_s": round(save_s, 3), "save_gbs": round(nbytes / save_s / 1e9, 2),
                      "restore_s": round(load_s, 3),
                      "restore_gbs": round(nbytes / load_s / 1e9, 2),
                      "restored_bitwise": bool(same),
                      "timing": "wall clock around each call, each ending synchronised"}),
          flush=True)


def bench_sweep(args):
    """The size sweep of the collectives (one process; each point the mean of
    back-to-back launches between one CUDA-event pair)."""
    import torch
    from gradient_sync_rcc_gb300 import build, rcc, synth
    build.build()
    dev = "cuda:0"
    peak, src = peak_hbm()
    sizes = [257 * 4 ** k for k in range(10)] + [1 << 28]
    for Rk in (2, 4, 8):
        for n in sizes:
            for case, dt in (("all_reduce_mean", rcc.F32), ("all_reduce_mean", rcc.BF16),
                             ("broadcast", rcc.F32), ("reduce", rcc.F32)):
                td = torch.float32 if dt == rcc.F32 else torch.bfloat16
                es = 4 if dt == rcc.F32 else 2
                ins = synth.gpu_rank_buffers("uniform", Rk, n, td, (5, Rk, n), dev)
                outs = [torch.empty(n, dtype=td, device=dev) for _ in range(Rk)]
                h = rcc.register(0, Rk, dt, True)
                try:
                    if case == "all_reduce_mean":
                        fn = lambda: rcc.all_reduce(h, ins, outs, "mean")
                        traffic = 2 * Rk * n * es
                    elif case == "broadcast":
                        fn = lambda: rcc.broadcast(h, ins[0], outs, root=0)
                        traffic = (Rk + 1) * n * es
                    else:
                        fn = lambda: rcc.reduce(h, ins, outs[Rk - 1], root=Rk - 1, op="mean")
                        traffic = (Rk + 1) * n * es
                    reps = 50 if traffic < (1 << 30) else 10
                    ms = timed_batch(torch, fn, reps)
                finally:
                    rcc.finish(h)
                gbs = traffic / (ms * 1e-3) / 1e9
                print(json.dumps({"sweep": case, "ranks": Rk, "elems": n,
                                  "dtype": "f32" if dt == rcc.F32 else "bf16",
                                  "ms": round(ms, 5), "timing": "%d back to back" % reps,
                                  "algbw_gbs": round(Rk * n * es / (ms * 1e-3) / 1e9, 1),
                                  "traffic_gbs": round(gbs, 1),
                                  "frac_of_" + src: round(gbs / peak, 4),
                                  "l2_resident": traffic < 129e6}), flush=True)
                del ins, outs
        torch.cuda.empty_cache()


def main():
    args = parse_args()
    if args.sweep:
        bench_sweep(args)
        return
    if args.case == "grad_sync_1024":
        bench_grad_sync_1024(args)
        return
    if args.case == "all_reduce_rank":
        bench_rank_case(args)
        return
    if args.case == "checkpoint":
        bench_checkpoint(args)
        return
    if args.case != "step":
        bench_case(args)
        return
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
