#!/usr/bin/env python3
"""Benchmark: implicit-GEMM conv2d forward on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one forward convolution of the workload (every hot-path stage runs
inside the one kernel launch).  The default workload is the 28x28 C256 ResNet
layer (GEMM 12544 x 256 x 2304), the largest compute-bound entry of the
benchmark list and the first one with a tensor-peak target.

``value`` is whole-job TFLOP/s (2*N*P*Q*K*C*R*S per step) with inputs resident
in HBM, device-timed with CUDA events around CUDA-graph replays of exactly K
launches.  Consecutive steps rotate through independent input/output buffer
sets (at least twice the L2 size in total), and the L2 is flushed by a 2 x L2
scratch write between the warm-up and the timed region, so no timed step finds
its inputs in L2 ("cold" mode).  ``hot_l2`` is the same K launches back to
back on one buffer set (inputs and output L2-resident after the first step).
``e2e`` is the same metric through the host-buffer entry point (pinned H2D
copies, kernel, D2H copy of y, every step).  ``--impl reference`` times the
CPU oracle on a bounded sample of the same workload instead.

Multi-GPU (torchrun): the convolution does not need an exchange step, so each
rank runs an independent replica on its own GPU (weak scaling); the job time is
the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "conv2d fwd TFLOP/s (2·NPQ·K·CRS/time) and % of GB300 BF16 tensor peak"
METRIC_WGRAD = "conv2d wgrad TFLOP/s (2·NPQ·K·CRS/time) and % of GB300 BF16 tensor peak"
METRIC_DGRAD = "conv2d dgrad TFLOP/s (2·NPQ·K·CRS/time) and % of GB300 BF16 tensor peak"
DEFAULT_WORKLOAD = "resnet_28x28_c256"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- workload arithmetic
def out_extent(in_size, pad, dil, ker, stride):
    span = dil * (ker - 1) + 1
    room = in_size + 2 * pad - span
    return 0 if room < 0 else room // stride + 1


def shape_of(wl):
    p = out_extent(wl.h, wl.pad_h, wl.dil_h, wl.r, wl.stride_h)
    q = out_extent(wl.w, wl.pad_w, wl.dil_w, wl.s, wl.stride_w)
    return p, q


def flops_per_step(wl):
    p, q = shape_of(wl)
    return 2.0 * wl.n * p * q * wl.k * (wl.c // wl.groups) * wl.r * wl.s


def _touched(extent_in, extent_out, stride, pad, dil, ker):
    rows = set()
    for o in range(extent_out):
        for t in range(ker):
            i = o * stride - pad + t * dil
            if 0 <= i < extent_in:
                rows.add(i)
    return len(rows)


def algorithmic_bytes(wl, out_bytes=4):
    """Input pixels some window touches (bf16) + weight (bf16) + output (fp32, or bf16 with
    the fused bf16-output epilogue) + bias (fp32)."""
    p, q = shape_of(wl)
    th = _touched(wl.h, p, wl.stride_h, wl.pad_h, wl.dil_h, wl.r)
    tw = _touched(wl.w, q, wl.stride_w, wl.pad_w, wl.dil_w, wl.s)
    x_b = wl.n * th * tw * wl.c * 2
    w_b = wl.k * wl.r * wl.s * (wl.c // wl.groups) * 2
    y_b = wl.n * p * q * wl.k * out_bytes
    b_b = wl.k * 4 if wl.bias is not None else 0
    return float(x_b + w_b + y_b + b_b)


def algorithmic_bytes_wgrad(wl):
    """Input pixels some window touches (bf16) + output gradient dy (bf16) + weight gradient (fp32)."""
    p, q = shape_of(wl)
    th = _touched(wl.h, p, wl.stride_h, wl.pad_h, wl.dil_h, wl.r)
    tw = _touched(wl.w, q, wl.stride_w, wl.pad_w, wl.dil_w, wl.s)
    return float(wl.n * th * tw * wl.c * 2 + wl.n * p * q * wl.k * 2 + wl.k * wl.r * wl.s * (wl.c // wl.groups) * 4)


def algorithmic_bytes_dgrad(wl):
    """Output gradient dy (bf16) + weights (bf16) + input gradient dx (fp32)."""
    p, q = shape_of(wl)
    return float(wl.n * p * q * wl.k * 2 + wl.k * wl.r * wl.s * wl.c * 2 + wl.n * wl.h * wl.w * wl.c * 4)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "split_gemm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    want = kernel_source_hash()
    for line in lines:
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == want:
            return float(parts[2])
    return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background; samples carry host timestamps."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu_index = gpu_index
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        where = "during"
        if not inside:  # timed region shorter than the sampling period: nearest samples after warm-up
            inside = [p for (t, p) in self.samples if t >= t0 - 0.5][:3]
            where = "adjacent"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = sorted(v for v in (num(p[1]) for p in inside) if v is not None)
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": where}


# ----------------------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist_mod, device=None):
    if dist_mod is not None:
        if device is not None and dist_mod.get_backend() == "nccl":
            dist_mod.barrier(device_ids=[device.index])
        else:
            dist_mod.barrier()


def aggregate(dist_mod, elapsed_s: float, units: float, device=None):
    """Job time = max over ranks; units = sum over ranks.  Returns (max_elapsed, total_units)."""
    if dist_mod is None:
        return elapsed_s, units
    import torch
    dev = device if (device is not None and dist_mod.get_backend() == "nccl") else torch.device("cpu")
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    dist_mod.all_reduce(u, op=dist_mod.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ----------------------------------------------------------------------------- CPU oracle sample
class OracleSampler:
    """Times the CPU oracle, as it stands, on bounded samples of the workload.

    Calibrated once on a single image.  A sample whose budget covers at least one
    whole image is the first ``nb`` images of the batch (all output channels,
    every host thread); a smaller budget gets randomly chosen output elements
    (one thread, inputs widened to float64 once up front).
    """

    def __init__(self, wl):
        import numpy as np

        import oracle
        self.oracle, self.np, self.wl = oracle, np, wl
        self.x, self.w, self.b = workloads.make_inputs(wl)
        self.opts = wl.options()
        self.threads = oracle.default_threads()
        self.lib = oracle.load()
        self.p, self.q = shape_of(wl)
        self.flop_img = flops_per_step(wl) / wl.n
        t0 = time.perf_counter()
        oracle.conv2d_fwd(self.x[:1], self.w, self.b, **self.opts, threads=self.threads, lib=self.lib)
        self.per_img = time.perf_counter() - t0
        self.xd = self.wd = None

    def run(self, budget_s: float):
        """One sample of about ``budget_s`` seconds: (TFLOP/s, threads, description, seconds)."""
        wl, oracle = self.wl, self.oracle
        if self.per_img <= budget_s:
            nb = max(1, min(wl.n, int(budget_s / self.per_img)))
            reps = 0
            t0 = time.perf_counter()
            while True:
                oracle.conv2d_fwd(self.x[:nb], self.w, self.b, **self.opts, threads=self.threads, lib=self.lib)
                reps += 1
                done = time.perf_counter() - t0
                if done + done / reps > budget_s or reps >= 1000:
                    break
            desc = f"{nb} of {wl.n} images x {reps} repetitions, {self.threads} threads"
            return self.flop_img * nb * reps / done / 1e12, self.threads, desc, done
        if self.xd is None:
            self.xd, self.wd = oracle.widen_bf16(self.x), oracle.widen_bf16(self.w)
        per_point = self.per_img * self.threads / (self.p * self.q * wl.k)
        npts = max(8, int(budget_s / per_point))
        rng = self.np.random.default_rng(npts)
        mi = rng.integers(0, wl.n * self.p * self.q, size=npts)
        ki = rng.integers(0, wl.k, size=npts)
        t0 = time.perf_counter()
        oracle.conv2d_fwd_points_f64(self.xd, self.wd, self.b, self.opts["stride"], self.opts["padding"],
                                     self.opts["dilation"], mi, ki, lib=self.lib, groups=self.opts["groups"])
        done = time.perf_counter() - t0
        flops = 2.0 * (wl.c // wl.groups) * wl.r * wl.s * npts
        return flops / done / 1e12, 1, f"{npts} random output elements, 1 thread", done


class WgradOracleSampler:
    """Times the weight-gradient oracle on randomly chosen gradient elements (one thread;
    inputs widened to float64 once): each element is a sum over the N*P*Q output pixels."""

    def __init__(self, wl):
        import numpy as np

        import oracle
        from oracle import wgrad as ow
        self.np, self.ow, self.wl = np, ow, wl
        x, w, _ = workloads.make_inputs(wl)
        dy = workloads.make_output_grad(wl)
        self.w_shape = tuple(w.shape)
        self.xd, self.dyd = oracle.widen_bf16(x), oracle.widen_bf16(dy)
        self.o = wl.options()
        self.lib = ow.load()
        self.L = dy.shape[0] * dy.shape[1] * dy.shape[2]
        self.cols = self.w_shape[1] * self.w_shape[2] * self.w_shape[3]
        t0 = time.perf_counter()
        self._points(8)
        self.per_point = max(1e-7, (time.perf_counter() - t0) / 8)

    def _points(self, npts):
        rng = self.np.random.default_rng(npts)
        kk = rng.integers(0, self.wl.k, size=npts)
        jj = rng.integers(0, self.cols, size=npts)
        self.ow.conv2d_wgrad_points_f64(self.xd, self.dyd, self.w_shape, self.o["stride"], self.o["padding"],
                                        self.o["dilation"], kk, jj, lib=self.lib)

    def run(self, budget_s: float):
        npts = max(8, int(budget_s / self.per_point))
        t0 = time.perf_counter()
        self._points(npts)
        done = time.perf_counter() - t0
        return 2.0 * self.L * npts / done / 1e12, 1, f"{npts} random weight-gradient elements, 1 thread", done


class DgradOracleSampler:
    """Times the data-gradient oracle on randomly chosen gradient elements (one thread)."""

    def __init__(self, wl):
        import numpy as np

        import oracle
        from oracle import dgrad as od
        self.np, self.od, self.wl = np, od, wl
        _, w, _ = workloads.make_inputs(wl)
        dy = workloads.make_output_grad(wl, variance=1.0)
        self.wd, self.dyd = oracle.widen_bf16(w), oracle.widen_bf16(dy)
        self.o = wl.options()
        self.lib = od.load()
        self.xs = (wl.n, wl.h, wl.w, wl.c)
        t0 = time.perf_counter()
        self._points(64)
        self.per_point = max(1e-7, (time.perf_counter() - t0) / 64)

    def _points(self, npts):
        rng = self.np.random.default_rng(npts)
        mi = rng.integers(0, self.wl.n * self.wl.h * self.wl.w, size=npts)
        ci = rng.integers(0, self.wl.c, size=npts)
        self.od.conv2d_dgrad_points_f64(self.dyd, self.wd, self.xs, self.o["stride"], self.o["padding"],
                                        self.o["dilation"], mi, ci, lib=self.lib)

    def run(self, budget_s: float):
        npts = max(64, int(budget_s / self.per_point))
        t0 = time.perf_counter()
        self._points(npts)
        done = time.perf_counter() - t0
        # Same FLOP count per step as the forward convolution, spread over N*H*W*C elements.
        flops = flops_per_step(self.wl) * npts / (self.wl.n * self.wl.h * self.wl.w * self.wl.c)
        return flops / done / 1e12, 1, f"{npts} random input-gradient elements, 1 thread", done


# ----------------------------------------------------------------------------- the GPU arm
def _sets_for(wl, set_bytes):
    return max(1, min(64, math.ceil(2 * L2_BYTES / max(1, set_bytes))))


def run_ours(args, wl, world, rank, local):
    import torch

    import split_gemm_gb300 as sg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_mod = init_dist(world, "nccl")
    sg.load_library()
    x, w, b = workloads.make_inputs(wl)
    params = sg.make_params(x.shape, w.shape, **wl.options())
    p, q = sg.output_shape(params)
    if args.op == "wgrad":
        return run_wgrad(args, wl, sg, torch, dev, dist_mod, x, w, params)
    if args.op == "dgrad":
        return run_dgrad(args, wl, sg, torch, dev, dist_mod, w, params)
    forced = _forced_algo(sg, args)
    relu, out_bf16 = args.epilogue in ("relu", "relu_bf16"), args.epilogue in ("bf16", "relu_bf16")
    y_dtype, y_bytes = (torch.bfloat16, 2) if out_bf16 else (torch.float32, 4)
    algo = sg.query_algo(params, relu=relu, out_bf16=out_bf16)
    if forced is not None:
        algo = _algo_report(algo, forced)
    set_bytes = x.numel() * 2 + w.numel() * 2 + wl.n * p * q * wl.k * y_bytes + (0 if b is None else b.numel() * 4)
    n_sets = _sets_for(wl, set_bytes)
    sets = []
    for _ in range(n_sets):
        sets.append((x.to(dev), w.to(dev), None if b is None else b.to(dev),
                     torch.empty((wl.n, p, q, wl.k), dtype=y_dtype, device=dev)))
    ws_need = sg.epi_workspace_bytes(params, forced, relu, out_bf16) if (relu or out_bf16) else sg.workspace_bytes(params)
    ws = torch.zeros(max(4096, ws_need), dtype=torch.uint8, device=dev)
    opts = wl.options()
    stream = torch.cuda.Stream(dev)

    def step(i):
        xd, wd, bd, yd = sets[i % n_sets]
        sg.conv2d_fwd_into(yd, xd, wd, bd, **opts, workspace=ws, algo=forced, relu=relu)

    def step_hot(i):
        xd, wd, bd, yd = sets[0]
        sg.conv2d_fwd_into(yd, xd, wd, bd, **opts, workspace=ws, algo=forced, relu=relu)

    def check():
        if sg.status(ws, stream) != 0:
            raise RuntimeError("device status reported a timeout during warm-up")

    K, W = args.steps, args.warmup
    elapsed, clocks, chunk = _time_graphs(torch, stream, step, K, W, n_sets, dev, dist_mod, check)
    launches = sg.last_launch_count()
    status = sg.status(ws, stream)
    flops = flops_per_step(wl)
    job_s, job_flops = aggregate(dist_mod, elapsed, flops * K, dev)
    hot = None
    if not args.no_hot:
        hot_s, _, _ = _time_graphs(torch, stream, step_hot, K, 0, 1, dev, dist_mod, check, flush=False, roll_s=0.05)
        hot_job_s, hot_flops = aggregate(dist_mod, hot_s, flops * K, dev)
        hot = {"value": hot_flops / hot_job_s / 1e12, "unit": "TFLOP/s", "ms_per_step": hot_job_s / K * 1e3,
               "mode": "hot: one buffer set, back to back (inputs and output L2-resident after the first step)"}
        status = status or sg.status(ws, stream)

    e2e = None
    if not args.no_e2e and args.epilogue == "none":
        e2e = run_e2e(sg, torch, dev, stream, wl, x, w, b, params, p, q, min(K, args.e2e_steps), dist_mod)
    return dict(elapsed=elapsed, job_s=job_s, job_flops=job_flops, algo=algo if isinstance(algo, dict) else algo.as_dict(), n_sets=n_sets,
                clocks=clocks, status=status, e2e=e2e, dist=dist_mod, graph_chunk=chunk,
                l2=_l2_statement(K, n_sets, set_bytes), hot=hot, launches_per_step=launches)


def _algo_report(heuristic, forced):
    """The configuration a line ran: the heuristic's, or the forced fields (0 = left to the
    heuristic) beside the heuristic's own choice, which a forced loader or tile may replace."""
    if forced is None:
        return heuristic.as_dict()
    return {"forced": {k: v for k, v in forced.as_dict().items() if v}, "heuristic": heuristic.as_dict()}


def _forced_algo(sg, args):
    if not (args.block_n or args.splits or args.loader or args.grid or args.block_m or args.reduction or args.pair_kb
            or args.tma_store):
        return None
    a = sg.Algo()
    a.block_n, a.splits, a.loader, a.grid = args.block_n, args.splits, args.loader, args.grid
    a.block_m, a.reduction = args.block_m, args.reduction
    a.debug_flags = {1: 2, 2: 4}.get(args.pair_kb, 0)  # CONV2D_DEBUG_PAIR_KB1 / KB2
    if args.tma_store:
        a.debug_flags |= sg.DEBUG_TMA_STORE
    return a


def _build_graphs(torch, stream, step, K, n_sets):
    """CUDA graphs of back-to-back launches covering K steps.  A graph's length is a multiple
    of the buffer-set count (or K itself when K < n_sets), so replaying one after another
    continues the rotation: the same set never comes round within n_sets consecutive steps."""
    chunk = min(K, 512)
    chunk = max(n_sets, (chunk // n_sets) * n_sets) if K >= n_sets else K
    full, rem = divmod(K, chunk)
    graphs = []
    for length in ([chunk] if full else []) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(length):
                step(i)
        graphs.append(g)
    plan = [graphs[0]] * full + ([graphs[-1]] if rem else [])
    with torch.cuda.stream(stream):  # one untimed replay of each graph (upload)
        for g in graphs:
            g.replay()
    stream.synchronize()
    return plan, chunk


def _time_graphs(torch, stream, step, K, W, n_sets, dev, dist_mod, check, flush=True, roll_s=0.25):
    """W warm-up steps, then exactly K steps replayed from CUDA graphs between two events.

    The clocks are sampled while the GPU runs these same launches: an untimed pre-roll of
    about ``roll_s`` seconds, the timed region, and a post-roll, all queued back to back on
    the stream (a timed region of a few hundred microseconds is far shorter than the
    sampling period).  With ``flush`` a 2 x L2 scratch write runs between the pre-roll and
    the timed region, so the timed steps start from an L2 that holds none of their inputs.
    Returns (seconds, clocks, chunk)."""
    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
    stream.synchronize()
    check()
    plan, chunk = _build_graphs(torch, stream, step, K, n_sets)
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    # Replays of the step graphs that fill about roll_s seconds (estimated from one timed pass).
    probe0, probe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        probe0.record(stream)
        for g in plan:
            g.replay()
        probe1.record(stream)
    stream.synchronize()
    pass_s = max(1e-6, probe0.elapsed_time(probe1) / 1e3)
    rolls = max(1, min(100000, int(roll_s / pass_s)))
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist_mod, dev)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        for _ in range(rolls):
            for g in plan:
                g.replay()
        if scratch is not None:
            scratch.fill_(1.0)
        start.record(stream)
        for g in plan:
            g.replay()
        end.record(stream)
        for _ in range(rolls):
            for g in plan:
                g.replay()
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(dist_mod, dev)
    clocks.stop()
    summary = clocks.summary(t0, t1)
    summary["window"] = ("pre-roll, timed region and post-roll of the same launches "
                         f"({rolls} untimed passes on each side)") if summary.get("window") == "during" else summary.get("window")
    return start.elapsed_time(end) / 1e3, summary, chunk


def _l2_statement(K, n_sets, set_bytes, flush=True):
    touched = min(K, n_sets)
    return {"mode": "cold: rotating buffer sets" + (", L2 flushed (2 x L2 write) before the timed region" if flush else ""),
            "buffer_sets": n_sets, "set_bytes": int(set_bytes), "sets_touched_in_timed_region": touched,
            "bytes_touched_in_timed_region": int(touched * set_bytes),
            "reuse_distance_bytes": int(n_sets * set_bytes) if K > n_sets else None}


def run_wgrad(args, wl, sg, torch, dev, dist_mod, x, w, params):
    """The weight gradient of the workload: conv2d_bwd_weight over rotating buffer sets."""
    dy = workloads.make_output_grad(wl)
    forced = _forced_algo(sg, args)
    algo = sg.query_wgrad_algo(params)
    if forced is not None:
        algo = _algo_report(algo, forced)
    set_bytes = x.numel() * 2 + dy.numel() * 2 + w.numel() * 4
    n_sets = _sets_for(wl, set_bytes)
    sets = [(x.to(dev), dy.to(dev), torch.empty(tuple(w.shape), dtype=torch.float32, device=dev))
            for _ in range(n_sets)]
    ws = torch.zeros(max(4096, sg.wgrad_workspace_bytes(params)), dtype=torch.uint8, device=dev)
    o = wl.options()
    opts = dict(stride=o["stride"], padding=o["padding"], dilation=o["dilation"])
    stream = torch.cuda.Stream(dev)

    def step(i):
        xd, dyd, dwd = sets[i % n_sets]
        sg.conv2d_bwd_weight_into(dwd, xd, dyd, **opts, workspace=ws, algo=forced)

    def check():
        if sg.status(ws, stream) != 0:
            raise RuntimeError("device status reported a timeout during warm-up")

    elapsed, clocks, chunk = _time_graphs(torch, stream, step, args.steps, args.warmup, n_sets, dev, dist_mod, check)
    launches = sg.last_launch_count()
    status = sg.status(ws, stream)
    flops = flops_per_step(wl)
    job_s, job_flops = aggregate(dist_mod, elapsed, flops * args.steps, dev)
    return dict(elapsed=elapsed, job_s=job_s, job_flops=job_flops, algo=algo if isinstance(algo, dict) else algo.as_dict(), n_sets=n_sets,
                clocks=clocks, status=status, e2e=None, dist=dist_mod, graph_chunk=chunk,
                l2=_l2_statement(args.steps, n_sets, set_bytes), hot=None, launches_per_step=launches)


def run_dgrad(args, wl, sg, torch, dev, dist_mod, w, params):
    """The data gradient of the workload: conv2d_bwd_data over rotating buffer sets."""
    dy = workloads.make_output_grad(wl, variance=1.0)
    forced = _forced_algo(sg, args)
    algo = sg.query_dgrad_algo(params)
    if forced is not None:
        algo = _algo_report(algo, forced)
    xs = (wl.n, wl.h, wl.w, wl.c)
    set_bytes = dy.numel() * 2 + w.numel() * 2 + wl.n * wl.h * wl.w * wl.c * 4
    n_sets = _sets_for(wl, set_bytes)
    sets = [(dy.to(dev), w.to(dev), torch.empty(xs, dtype=torch.float32, device=dev)) for _ in range(n_sets)]
    ws = torch.zeros(max(4096, sg.dgrad_workspace_bytes(params)), dtype=torch.uint8, device=dev)
    o = wl.options()
    opts = dict(stride=o["stride"], padding=o["padding"], dilation=o["dilation"])
    stream = torch.cuda.Stream(dev)

    def step(i):
        dyd, wd, dxd = sets[i % n_sets]
        sg.conv2d_bwd_data_into(dxd, dyd, wd, **opts, workspace=ws, algo=forced)

    def check():
        if sg.status(ws, stream) != 0:
            raise RuntimeError("device status reported a timeout during warm-up")

    elapsed, clocks, chunk = _time_graphs(torch, stream, step, args.steps, args.warmup, n_sets, dev, dist_mod, check)
    launches = sg.last_launch_count()
    status = sg.status(ws, stream)
    job_s, job_flops = aggregate(dist_mod, elapsed, flops_per_step(wl) * args.steps, dev)
    return dict(elapsed=elapsed, job_s=job_s, job_flops=job_flops, algo=algo if isinstance(algo, dict) else algo.as_dict(), n_sets=n_sets,
                clocks=clocks, status=status, e2e=None, dist=dist_mod, graph_chunk=chunk,
                l2=_l2_statement(args.steps, n_sets, set_bytes), hot=None, launches_per_step=launches)


def run_e2e(sg, torch, dev, stream, wl, x, w, b, params, p, q, steps, dist_mod):
    """Same metric through the host-buffer entry point: H2D of x, w, bias + kernel + D2H of y, every step.

    Steps alternate over two streams, each with its own device staging buffer and pinned output
    buffer, so one step's uploads can overlap the previous step's download (H2D and D2H run on
    separate copy engines), as a serving loop would pipeline requests.  The single-stream figure,
    where every step waits for the previous step's download, is reported beside it."""
    lanes = 2
    streams = [stream] + [torch.cuda.Stream(dev) for _ in range(lanes - 1)]
    staging = [torch.zeros(sg.host_staging_bytes(params), dtype=torch.uint8, device=dev) for _ in range(lanes)]
    xh, wh = x.pin_memory(), w.pin_memory()
    bh = None if b is None else b.pin_memory()
    yh = [torch.empty((wl.n, p, q, wl.k), dtype=torch.float32).pin_memory() for _ in range(lanes)]

    def timed(n_lanes):
        for i in range(3 * n_lanes):
            sg.conv2d_fwd_host(xh, wh, bh, yh[i % n_lanes], params, staging[i % n_lanes], streams[i % n_lanes])
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        done = [torch.cuda.Event() for _ in range(n_lanes)]
        end = torch.cuda.Event(enable_timing=True)
        barrier(dist_mod, dev)
        torch.cuda.synchronize()
        start.record(streams[0])
        for k in range(1, n_lanes):
            streams[k].wait_event(start)
        for i in range(steps):
            sg.conv2d_fwd_host(xh, wh, bh, yh[i % n_lanes], params, staging[i % n_lanes], streams[i % n_lanes])
        for k in range(1, n_lanes):
            done[k].record(streams[k])
            streams[0].wait_event(done[k])
        end.record(streams[0])
        torch.cuda.synchronize()
        return aggregate(dist_mod, start.elapsed_time(end) / 1e3, flops_per_step(wl) * steps, dev)

    serial_s, serial_flops = timed(1)
    job_s, job_flops = timed(lanes)
    h2d = x.numel() * 2 + w.numel() * 2 + (0 if b is None else b.numel() * 4)
    return {"value": job_flops / job_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(wl.n * p * q * wl.k * 4), "steps": steps,
            "ms_per_step": job_s / steps * 1e3, "streams": lanes,
            "serial": {"value": serial_flops / serial_s / 1e12, "ms_per_step": serial_s / steps * 1e3}}


# ----------------------------------------------------------------------------- JSON assembly
def config_of(wl, extra=None):
    p, q = shape_of(wl)
    cfg = {"workload": wl.name, "shape": wl.describe(), "gemm_mnk": [wl.n * p * q, wl.k, wl.c * wl.r * wl.s],
           "bias": wl.bias is not None, "layout": "x NHWC bf16, w KRSC bf16, bias fp32, y NHWC fp32"}
    if extra:
        cfg.update(extra)
    return cfg


def roofline(wl, t_step_s, peaks, peak_src, out_bytes=4, op="fwd"):
    flops = flops_per_step(wl)
    nbytes = (algorithmic_bytes_wgrad(wl) if op == "wgrad" else algorithmic_bytes_dgrad(wl) if op == "dgrad"
              else algorithmic_bytes(wl, out_bytes))
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    traffic = recorded_traffic(wl.name if op == "fwd" else f"{wl.name}:{op}") if out_bytes == 4 else None
    note = ("dram__bytes_read.sum + dram__bytes_write.sum of one launch captured alone under ncu "
            "(profiles/ncu_traffic.txt): inputs read from DRAM once; an output smaller than L2 is still in L2 "
            "when the launch ends, so its write-back is not in the figure") if traffic is not None else None
    if flops / nbytes >= ridge:
        achieved = flops / t_step_s / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "peak_source": f"{peak_src} (bf16 burst)", "traffic": traffic, "traffic_source": note,
                "algorithmic_bytes": nbytes,
                "algorithmic_flops": flops}
    achieved = nbytes / t_step_s / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peak_src} (HBM copy)", "traffic": traffic,
            "traffic_source": note,
            "algorithmic_bytes": nbytes, "algorithmic_flops": flops}


def main_ours(args):
    wl = workloads.get(args.workload)
    world, rank, local = dist_env()
    res = run_ours(args, wl, world, rank, local)
    peaks, peak_src = load_peaks()
    K = args.steps
    t_step = res["elapsed"] / K
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        sampler = {"wgrad": WgradOracleSampler, "dgrad": DgradOracleSampler}.get(args.op, OracleSampler)(wl)
        v, cores, desc, secs = sampler.run(args.cpu_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               "seconds": round(secs, 2)}
    if res["dist"] is not None:
        res["dist"].destroy_process_group()
    if rank != 0:
        return 0
    value = res["job_flops"] / res["job_s"] / 1e12
    line = {
        "metric": {"wgrad": METRIC_WGRAD, "dgrad": METRIC_DGRAD}.get(args.op, METRIC), "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup,
        "ms_per_step": res["job_s"] / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_of(wl, {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                 "algo": res["algo"], "accumulate": "fp32 (TMEM)",
                                 "epilogue": {"none": "bias, fp32 y", "relu": "bias, ReLU, fp32 y",
                                              "bf16": "bias, bf16 y", "relu_bf16": "bias, ReLU, bf16 y"}[args.epilogue],
                                 **({"layout": "x NHWC bf16, w KRSC bf16, bias fp32, y NHWC bf16"}
                                    if args.epilogue in ("bf16", "relu_bf16") else {}),
                                 **({"op": "weight gradient", "epilogue": "fp32 dw",
                                     "layout": "x NHWC bf16, dy NPQK bf16 ~N(0, 2/(N*P*Q)), dw KRSC fp32",
                                     "gemm_mnk": [wl.k, wl.r * wl.s * wl.c, wl.n * shape_of(wl)[0] * shape_of(wl)[1]]}
                                    if args.op == "wgrad" else {}),
                                 **({"op": "data gradient", "epilogue": "fp32 dx",
                                     "layout": "dy NPQK bf16 ~N(0, 1), w KRSC bf16, dx NHWC fp32",
                                     "gemm_mnk": [wl.n * wl.h * wl.w, wl.c, wl.k * wl.r * wl.s]}
                                    if args.op == "dgrad" else {}),
                                 "l2": res["l2"],
                                 "timing": f"CUDA events around CUDA-graph replays ({res['graph_chunk']} launches "
                                           "per graph), max over ranks"}),
        "roofline": roofline(wl, t_step, peaks, peak_src, 2 if args.epilogue in ("bf16", "relu_bf16") else 4, args.op),
        "hot_l2": res["hot"],
        "cpu_baseline": cpu,
        "e2e": res["e2e"],
        "gpu_launches": K * max(1, res["launches_per_step"]),
        "clocks": res["clocks"],
        "device_status": res["status"],
    }
    print(json.dumps(line), flush=True)
    return 0 if res["status"] == 0 else 1


def main_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded sample of the same workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = workloads.get(args.workload)
    sampler = {"wgrad": WgradOracleSampler, "dgrad": DgradOracleSampler}.get(args.op, OracleSampler)(wl)
    per_step = max(0.001, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        sampler.run(per_step)
    vals, cores, desc, total = [], 1, "", 0.0
    for _ in range(args.steps):
        v, cores, desc, secs = sampler.run(per_step)
        vals.append(v)
        total += secs
    value = sum(vals) / len(vals) if vals else 0.0
    line = {
        "impl": "reference", "metric": {"wgrad": METRIC_WGRAD, "dgrad": METRIC_DGRAD}.get(args.op, METRIC),
        "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, {"parallelism": "CPU oracle, rank 0 only"}),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-hot", action="store_true", help="skip the hot-L2 (one buffer set) timing")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of CPU oracle time for cpu_baseline")
    ap.add_argument("--block-n", type=int, default=0, help="force the output-channel tile width (64/128/256)")
    ap.add_argument("--splits", type=int, default=0, help="force the split-K factor")
    ap.add_argument("--reduction", type=int, default=0,
                    help="force the in-place reduction of cut tiles (1 ordered, 2 concurrent)")
    ap.add_argument("--loader", type=int, default=0, help="force the im2col loader (1 TMA, 2 cp.async, 3 scalar, 4 hybrid, 5 row window, 6 TMA box, 7 halo)")
    ap.add_argument("--grid", type=int, default=0, help="force the number of CTAs sharing the work (stream-K)")
    ap.add_argument("--block-m", type=int, default=0, help="force the output-pixel tile height (128/256)")
    ap.add_argument("--pair-kb", type=int, default=0, choices=[0, 1, 2],
                    help="CTA-pair loader: force 1 or 2 k-blocks per pipeline stage (0: the heuristic's)")
    ap.add_argument("--tma-store", action="store_true",
                    help="CTA-pair loaders: write y through TMA stores (a measurement hook)")
    ap.add_argument("--op", default="fwd", choices=["fwd", "wgrad", "dgrad"],
                    help="fwd: the forward convolution (the headline); wgrad / dgrad: its weight / input gradient")
    ap.add_argument("--epilogue", default="none", choices=["none", "relu", "bf16", "relu_bf16"],
                    help="fused epilogue variant (ReLU after the bias, bf16 output); the e2e leg runs only for none")
    args = ap.parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    return args


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return main_reference(args)
    return main_ours(args)


if __name__ == "__main__":
    sys.exit(main())
