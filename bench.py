#!/usr/bin/env python
"""Benchmark of the MX block-scaled NT GEMM on GB300.

Default line: the 4096^3 MXFP8 workload (E4M3 codes from N(0,1), E8M0 scale per
32 along K, BF16 out).  One step = the whole per-call hot path on one batch:
  mxgemm_prepare + mxgemm_run  -> C from A, row-major SA, B and the weight's
                                  tile-layout SB.  The activation scales (SA) are
                                  laid out inside the GEMM kernel for this plan
                                  ("sa=in-kernel": one launch per step); plans
                                  that cannot do that launch a relayout first.
The weight's scales (SB) are laid out once per weight, before the timed region.
The K steps are timed twice, as stream launches and as one CUDA-graph replay;
the headline takes the faster, and both are in the line.
Inputs are resident in HBM when the timed region starts; the step rotates over
enough input/output sets that their total exceeds twice the L2, so no step
reads another step's data from L2.  `e2e` repeats the step through mxgemm_run
from pinned HOST buffers, with the copies in the timed region.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--sweep]

With --gpus N under torchrun every rank runs an independent replica (the GEMM
has no exchange step); value = all ranks' FLOPs / the slowest rank's time.
--impl reference times the CPU oracle (the only other program computing the
same result here) on a bounded sample of the same workload.
--sweep prints one line per shape of the model workloads (not the headline);
--quant-sweep one line per activation shape for the MX quantiser; --grouped-sweep
one line per grouped (mixture-of-experts) case; --tensor-probe one line per MMA
kind and tile of the tensor pipe's own rate (operands resident in shared memory),
the ceiling the GEMM lines are compared with.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4/MXFP8 NT GEMM TFLOP/s on 1 GB300; % of dense MX tensor (or HBM) roofline"
WORKLOAD = "mxfp8_square_4096"
NOMINAL_PF = {"bf16": 2.25, "mxfp8": 4.5, "mxfp4": 13.5}
# the GEMM kernels and the host code that plans them (tile, stream-K split)
KERNEL_SOURCES = ["mx_block_scaled_gb300/csrc/gemm_kernel.cuh", "mx_block_scaled_gb300/csrc/ptx.cuh",
                  "mx_block_scaled_gb300/csrc/gemm_fp8.cu", "mx_block_scaled_gb300/csrc/gemm_fp4.cu",
                  "mx_block_scaled_gb300/csrc/gemm_kernel_pair.cuh", "mx_block_scaled_gb300/csrc/mxgemm.cu",
                  "mx_block_scaled_gb300/csrc/launch_impl.cuh", "mx_block_scaled_gb300/csrc/launch.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")


# ----------------------------------------------------------------- helpers --

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def slowest_rank_ms(ms: float, ws: int, device) -> float:
    """Replicas: every rank times the same work; the job's time is the slowest
    rank's (all_reduce MAX over the default process group when ws > 1)."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def versions() -> dict:
    """Library, CUDA, driver, PyTorch and numpy versions of the run and the hash of the
    kernel sources (recorded beside the plan; a copy of the sources may carry no git history)."""
    import numpy
    import torch
    out = {"torch": torch.__version__, "numpy": numpy.__version__, "cuda_runtime": torch.version.cuda,
           "kernel_source_sha": kernel_source_sha()}
    try:
        from mx_block_scaled_gb300 import binding as mx
        out["libmxgemm"] = int(mx.mxgemm_version())
    except Exception:  # the line is still useful without it
        pass
    try:
        q = subprocess.run(["nvidia-smi", "--query-gpu=driver_version,name", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=10).stdout.strip().splitlines()
        if q:
            drv, name = (x.strip() for x in q[0].split(",", 1))
            out.update(driver=drv, gpu=name)
    except (OSError, subprocess.SubprocessError, ValueError):
        pass
    return out


def job_tflops(flops_per_rank_step: float, ws: int, ms_per_step: float) -> float:
    """Whole-job throughput: all ranks' FLOPs over the slowest rank's step time."""
    return flops_per_rank_step * ws / (ms_per_step / 1e3) / 1e12


def kernel_source_sha() -> str:
    """Hash of the kernel and planner sources with comments and whitespace removed,
    so that a comment edit does not orphan a DRAM-traffic capture of the same code."""
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)  # block comments
        text = re.sub(r"//[^\n]*", " ", text)                 # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def mx_peak_tflops(fmt_name: str, bf16_tflops: float) -> float:
    return bf16_tflops * NOMINAL_PF[fmt_name] / NOMINAL_PF["bf16"]


def algorithmic_bytes(M, N, K, fmt_name, out_bytes):
    e = 1.0 if fmt_name == "mxfp8" else 0.5
    return (M + N) * K * e + (M + N) * K / 32 + M * N * out_bytes


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons (200 ms)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(loaded), "power_w_max": max(power)}


def read_traffic(fmt_name, M, N, K):
    """DRAM bytes per GEMM launch from a committed ncu capture, if the kernel sources still match."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    ent = d.get(f"{fmt_name}_{M}x{N}x{K}")
    if not ent or ent.get("kernel_source_sha") != kernel_source_sha():
        return None, None
    return ent.get("dram_bytes_per_launch"), ent.get("note")


# ----------------------------------------------------------- reference arm --

def oracle_sample_time(A, SA, B, SB, K, fmt, target_s: float, rows_cap: int):
    """Time the CPU oracle on the first r rows of C, r grown until one call takes
    about target_s.  Returns (rows, seconds, threads)."""
    import numpy as np
    import oracle
    oracle.build()
    rows = 8
    while True:
        idx = np.arange(rows, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.gemm(fmt, A, SA, B, SB, K, rows=idx, with_abs=False)
        dt = time.perf_counter() - t0
        if dt >= target_s or rows >= rows_cap:
            return rows, dt, oracle.num_threads()
        grow = max(2.0, min(16.0, target_s / max(dt, 1e-3)))
        rows = min(rows_cap, int(rows * grow))


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    from mx_block_scaled_gb300.inputs import FMT_MXFP8, make_operand
    M = N = K = 4096
    A, SA = make_operand(WORKLOAD, "A", 0, M, K, FMT_MXFP8)
    B, SB = make_operand(WORKLOAD, "B", 0, N, K, FMT_MXFP8)
    # size one step so that warmup + steps finish within a few minutes
    budget_s = 150.0 / max(1, args.steps + args.warmup)
    rows, _, threads = oracle_sample_time(A, SA, B, SB, K, 1, min(10.0, budget_s), M)
    import oracle
    idx = np.arange(rows, dtype=np.int64)
    for _ in range(args.warmup):
        oracle.gemm(1, A, SA, B, SB, K, rows=idx, with_abs=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm(1, A, SA, B, SB, K, rows=idx, with_abs=False)
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows * N * K / dt / 1e12
    sample = f"rows 0..{rows - 1} of C ({rows}x{N}x{K} of the {M}x{N}x{K} product) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "mxfp8 NT GEMM M=N=K=4096, E4M3 from N(0,1), E8M0/32, BF16 out",
                   "M": M, "N": N, "K": K, "format": "mxfp8", "out": "bf16"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- our arm --

# Further workload shapes timed in the same run as the headline line, so that one
# driver-run record carries both formats and both bounds: the 70B gate+up
# projection at prefill (M = 16384 tokens) in MXFP8 and MXFP4, and the same
# weight at decode (M = 8 tokens, weight-streaming, HBM-bound).
EXTRA_SHAPES = [("llama33_70b gate+up prefill", "mxfp8", 16384, 57344, 8192),
                ("llama33_70b gate+up prefill", "mxfp4", 16384, 57344, 8192),
                ("llama33_70b gate+up decode", "mxfp8", 8, 57344, 8192)]


def time_shape(mx, dev, fmt_name, M, N, K, reps, warmup=3, seed=0):
    """GEMM time of one shape through mxgemm_run (scales pre-laid-out, as a
    weight's are after loading and an activation's after the quantiser writes
    them in the tile layout): device-side random codes (E4M3 NaN codes
    excluded) and scale codes 120..134, rotating input/output sets whose total
    exceeds twice the L2; `reps` back-to-back calls between CUDA events on the
    launching stream, after `warmup` calls.  Returns (us per call, plan text,
    number of input sets)."""
    import torch
    from mx_block_scaled_gb300.inputs import FMT_BY_NAME
    fmt = FMT_BY_NAME[fmt_name]
    rb = K if fmt_name == "mxfp8" else K // 2
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = (M + N) * rb + (M + N) * K // 32 + M * N * 2
    nsets = max(2, math.ceil(2 * l2 / set_bytes) + 1)
    nsets = min(nsets, max(2, int(40e9 // set_bytes)))
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def codes(rows):
        c = torch.randint(0, 256, (rows, rb), dtype=torch.uint8, device=dev, generator=g)
        if fmt_name == "mxfp8":
            c = torch.where((c & 0x7F) == 0x7F, c & 0xFE, c)
        return c

    plan = mx.Plan(M, N, K, fmt, mx.MXGEMM_OUT_BF16, device=dev)
    sets = []
    for _ in range(nsets):
        SA = torch.randint(120, 135, (M, K // 32), dtype=torch.uint8, device=dev, generator=g)
        SB = torch.randint(120, 135, (N, K // 32), dtype=torch.uint8, device=dev, generator=g)
        sets.append((codes(M), mx.relayout_scales(SA, M, K), codes(N), mx.relayout_scales(SB, N, K),
                     torch.empty((M, N), dtype=torch.bfloat16, device=dev)))
        del SA, SB
    # weights are only read: MXGEMM_RUN_B_STATIC lets the decode plans start
    # loading them before the preceding call has finished
    pre = mx.MXGEMM_RUN_SA_PRELAYOUT | mx.MXGEMM_RUN_SB_PRELAYOUT | mx.MXGEMM_RUN_B_STATIC

    def one(i):
        a, sa, b, sb, c = sets[i % nsets]
        st = mx.mxgemm_run(plan.handle, a.data_ptr(), sa.data_ptr(), b.data_ptr(), sb.data_ptr(), c.data_ptr(),
                           plan.workspace.data_ptr(), plan.ws_bytes, pre, stream.cuda_stream)
        assert st == 0, mx.mxgemm_status_str(st)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(reps):
        one(i)
    e1.record(stream)
    torch.cuda.synchronize()
    mx.check_device_status()
    us = e0.elapsed_time(e1) * 1e3 / reps
    desc = plan.describe()
    del sets, plan
    torch.cuda.empty_cache()
    return us, desc, nsets


def extra_shape_record(label, fmt_name, M, N, K, us, desc, nsets, hbm_gbs, bf16_tf, peak_src):
    """One timed shape as a JSON object: TFLOP/s, GB/s and the roofline of its
    bound (the slower of the MX tensor peak and the algorithmic bytes over the
    measured HBM bandwidth)."""
    flops = 2.0 * M * N * K
    byts = algorithmic_bytes(M, N, K, fmt_name, 2)
    peak = mx_peak_tflops(fmt_name, bf16_tf)
    t = us / 1e6
    tensor_bound = flops / (peak * 1e12) > byts / (hbm_gbs * 1e9)
    tflops, gbs = flops / t / 1e12, byts / t / 1e9
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                "peak_source": f"{peak_src} bf16 burst {bf16_tf} TFLOP/s x nominal {fmt_name}/bf16 ratio "
                               f"{NOMINAL_PF[fmt_name] / NOMINAL_PF['bf16']:g}"}
    else:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs,
                "algorithmic_bytes": byts, "peak_source": f"{peak_src} HBM copy bandwidth"}
    return {"workload": f"{label}: {fmt_name} NT GEMM M={M} N={N} K={K}, BF16 out", "format": fmt_name,
            "M": M, "N": N, "K": K, "us": us, "tflops": tflops, "gbs": gbs, "roofline": roof, "plan": desc,
            "data": f"device-side random codes, scales 120..134, pre-laid-out; {nsets} rotating sets > 2x L2"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    from mx_block_scaled_gb300 import binding as mx
    from mx_block_scaled_gb300.inputs import FMT_MXFP8, make_operand

    fmt_name, fmt = "mxfp8", FMT_MXFP8
    M = N = K = 4096
    out_bytes = 2
    A, SA = make_operand(WORKLOAD, "A", 0, M, K, fmt)
    B, SB = make_operand(WORKLOAD, "B", 0, N, K, fmt)

    plan = mx.Plan(M, N, K, fmt, mx.MXGEMM_OUT_BF16, device=dev)
    desc = plan.describe()
    split = int(desc.split("split_k=")[1].split()[0])

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = A.nbytes + B.nbytes + SA.nbytes + SB.nbytes + M * N * out_bytes + mx.mxgemm_sf_bytes(N, K)
    nsets = max(3, math.ceil(2 * l2 / set_bytes) + 1)
    sets = []
    for _ in range(nsets):
        sets.append({
            "A": torch.from_numpy(A).to(dev), "B": torch.from_numpy(B).to(dev),
            "SA": torch.from_numpy(SA).to(dev), "SB": torch.from_numpy(SB).to(dev),
            "tSB": torch.empty(mx.mxgemm_sf_bytes(N, K), dtype=torch.uint8, device=dev),
            "C": torch.empty((M, N), dtype=torch.bfloat16, device=dev),
        })
    # step (1), mxgemm_prepare: SA relayout into the plan's workspace (+ stream-K
    # counter reset); step (2), mxgemm_run on the prepared workspace: the GEMM
    pre = mx.MXGEMM_RUN_SB_PRELAYOUT
    # The weight's scales (SB) are laid out once, when the weight is loaded (like
    # its quantisation); every call lays out the activation scales (SA).
    for s in sets:
        assert mx.mxgemm_relayout_scales(s["SB"].data_ptr(), N, K, s["tSB"].data_ptr(), sh) == 0
    torch.cuda.synchronize()

    launch = {"sh": sh}  # the stream the steps launch on (a side stream while a graph is captured)

    def step(i, ev=None):
        sh = launch["sh"]
        s = sets[i % nsets]
        if ev is not None:
            ev[0].record(stream)
        st = mx.mxgemm_prepare(plan.handle, s["SA"].data_ptr(), 0, plan.workspace.data_ptr(), plan.ws_bytes, pre,
                               sh)
        assert st == 0, mx.mxgemm_status_str(st)
        if ev is not None:
            ev[1].record(stream)
        st = mx.mxgemm_run(plan.handle, s["A"].data_ptr(), s["SA"].data_ptr(), s["B"].data_ptr(),
                           s["tSB"].data_ptr(), s["C"].data_ptr(), plan.workspace.data_ptr(), plan.ws_bytes,
                           pre | mx.MXGEMM_RUN_PREPARED, sh)
        assert st == 0, mx.mxgemm_status_str(st)
        if ev is not None:
            ev[2].record(stream)

    # in timed region 1: the SA relayout (unless the GEMM lays SA out itself), the
    # GEMM, and a split-K reduce
    sa_in_kernel = "sa=in-kernel" in desc
    launches_per_step = (0 if sa_in_kernel else 1) + 1 + (1 if split > 1 else 0)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    mx.check_device_status()

    sampler = ClockSampler(local)
    sampler.start()
    # clock soak: the same steps, untimed, long enough for nvidia-smi to see the load
    t_soak = time.perf_counter()
    i = 0
    while time.perf_counter() - t_soak < args.soak_s:
        for _ in range(20):
            step(i)
            i += 1
        torch.cuda.synchronize()

    # Timed region 1 -- the headline: K steps back to back with an event only at
    # each end, so that every GEMM launch may start its prologue while the
    # relayout before it finishes (programmatic dependent launch).
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    t_start.record(stream)
    for k in range(args.steps):
        step(k)
    t_end.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    wall_s = time.perf_counter() - w0
    stream_total_ms = t_start.elapsed_time(t_end)
    # Timed region 1b -- the same K steps captured once into a CUDA graph and
    # replayed (how a serving loop launches them: no per-launch host work between
    # the kernels, programmatic-dependent-launch edges kept in the graph).  The
    # headline is the faster of the two launch modes; both are reported.
    capture = torch.cuda.Stream(device=dev)  # graphs are captured off the default stream
    graph = torch.cuda.CUDAGraph()
    launch["sh"] = capture.cuda_stream
    with torch.cuda.graph(graph, stream=capture):
        for k in range(args.steps):
            step(k)
    launch["sh"] = sh
    graph.replay()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    r_start, r_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r_start.record(stream)
    graph.replay()
    r_end.record(stream)
    torch.cuda.synchronize()
    graph_total_ms = r_start.elapsed_time(r_end)
    total_ms = min(stream_total_ms, graph_total_ms)
    launch_mode = "cuda-graph replay" if graph_total_ms <= stream_total_ms else "stream launches"
    # Timed region 2 -- the GEMM kernel's own duration (roofline): K GEMM launches
    # back to back on the prepared workspace of each rotating set, events only at
    # the ends (the kernel's average duration as a stream runs it).
    def gemm_only(i):
        sh = launch["sh"]
        s = sets[i % nsets]
        st = mx.mxgemm_run(plan.handle, s["A"].data_ptr(), s["SA"].data_ptr(), s["B"].data_ptr(),
                           s["tSB"].data_ptr(), s["C"].data_ptr(), plan.workspace.data_ptr(), plan.ws_bytes,
                           pre | mx.MXGEMM_RUN_PREPARED, sh)
        assert st == 0, mx.mxgemm_status_str(st)

    torch.cuda.synchronize()
    g_start, g_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g_start.record(stream)
    for k in range(args.steps):
        gemm_only(k)
    g_end.record(stream)
    torch.cuda.synchronize()
    gemm_graph = torch.cuda.CUDAGraph()
    launch["sh"] = capture.cuda_stream
    with torch.cuda.graph(gemm_graph, stream=capture):
        for k in range(args.steps):
            gemm_only(k)
    launch["sh"] = sh
    gemm_graph.replay()
    torch.cuda.synchronize()
    gg_start, gg_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gg_start.record(stream)
    gemm_graph.replay()
    gg_end.record(stream)
    # Timed region 3 -- the same K steps with an event around each launch (the
    # relayout's own time; the events serialise the launches).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        step(k, evs[k])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    mx.check_device_status()

    gemm_stream_ms = g_start.elapsed_time(g_end) / args.steps
    gemm_graph_ms = gg_start.elapsed_time(gg_end) / args.steps
    gemm_ms = [min(gemm_stream_ms, gemm_graph_ms)]
    gemm_bracketed_ms = [e[1].elapsed_time(e[2]) for e in evs]
    relayout_ms = [e[0].elapsed_time(e[1]) for e in evs]
    serialised_ms = evs[0][0].elapsed_time(evs[-1][2]) / args.steps
    ms_per_step = slowest_rank_ms(total_ms / args.steps, ws, dev)
    flops = 2.0 * M * N * K
    value = job_tflops(flops, ws, ms_per_step)

    # ---- e2e: pinned host inputs -> device -> mxgemm_run (relayout + GEMM) -> host C.
    # Every step copies its inputs in and its result out inside the timed region.
    # Pipelined as a serving loop runs it: copy-in, compute and copy-out streams
    # over two device buffer sets, so that step i+1's upload and step i-1's
    # download overlap step i's GEMM (a second copy-in stream measured no
    # faster: the uploads are bound by the host link).  The one-stream (serial)
    # figure is kept too.
    e2e = None
    if not args.no_e2e:
        hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
        hSA, hSB = torch.from_numpy(SA).pin_memory(), torch.from_numpy(SB).pin_memory()
        hC = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        bufs = [sets[0], sets[1 % nsets]]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        done_cmp = [torch.cuda.Event() for _ in range(2)]
        done_out = [torch.cuda.Event() for _ in range(2)]
        done_in = [torch.cuda.Event() for _ in range(2)]

        def run_gemm(d, strm):
            st = mx.mxgemm_run(plan.handle, d["A"].data_ptr(), d["SA"].data_ptr(), d["B"].data_ptr(),
                               d["SB"].data_ptr(), d["C"].data_ptr(), plan.workspace.data_ptr(), plan.ws_bytes,
                               0, strm.cuda_stream)
            assert st == 0

        def e2e_step_serial():
            d = bufs[0]
            d["A"].copy_(hA, non_blocking=True)
            d["SA"].copy_(hSA, non_blocking=True)
            d["B"].copy_(hB, non_blocking=True)
            d["SB"].copy_(hSB, non_blocking=True)
            run_gemm(d, stream)
            hC[0].copy_(d["C"], non_blocking=True)

        def e2e_step_pipelined(i):
            b = i % 2
            d = bufs[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(done_cmp[b])  # step i-2's GEMM has read these inputs
                d["A"].copy_(hA, non_blocking=True)
                d["SA"].copy_(hSA, non_blocking=True)
                d["B"].copy_(hB, non_blocking=True)
                d["SB"].copy_(hSB, non_blocking=True)
                done_in[b].record(s_in)
            stream.wait_event(done_in[b])
            stream.wait_event(done_out[b])  # step i-2's result has been read out of C
            run_gemm(d, stream)
            done_cmp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_cmp[b])
                hC[b].copy_(d["C"], non_blocking=True)
                done_out[b].record(s_out)

        # a serving loop runs many steps: time up to 50 so that the pipeline's
        # fill and drain (one upload, one download) weigh little
        n_e2e = max(5, min(args.steps, 50))

        def timed(fn, pipelined):
            for i in range(3):
                fn(i) if pipelined else fn()
            torch.cuda.synchronize()
            if ws > 1:
                dist.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            s_in.wait_event(e0)
            s_out.wait_event(e0)
            for i in range(n_e2e):
                fn(i) if pipelined else fn()
            if pipelined:
                stream.wait_stream(s_out)
            e1.record(stream)
            torch.cuda.synchronize()
            return slowest_rank_ms(e0.elapsed_time(e1) / n_e2e, ws, dev)

        serial_ms = timed(e2e_step_serial, False)
        e2e_ms = timed(e2e_step_pipelined, True)
        mx.check_device_status()

        # The host link's own rates for the same tensors (one direction alone,
        # then both at once), which bound the pipelined step from below.
        def link_ms(fn, reps=5):
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        def up():
            bufs[0]["A"].copy_(hA, non_blocking=True)
            bufs[0]["B"].copy_(hB, non_blocking=True)

        def down():
            hC[0].copy_(bufs[1]["C"], non_blocking=True)

        def both():
            ev = torch.cuda.Event()
            ev.record(stream)
            s_out.wait_event(ev)
            up()
            with torch.cuda.stream(s_out):
                down()
            stream.wait_stream(s_out)

        up_b, down_b = A.nbytes + B.nbytes, M * N * out_bytes
        up_ms, down_ms, both_ms = link_ms(up), link_ms(down), link_ms(both)
        h2d_b = A.nbytes + B.nbytes + SA.nbytes + SB.nbytes
        link = {"h2d_gbs": up_b / up_ms / 1e6, "d2h_gbs": down_b / down_ms / 1e6,
                "both_dirs_ms": both_ms,
                "bound_ms_per_step": both_ms * h2d_b / up_b}  # + the scales' upload
        e2e = {"value": job_tflops(flops, ws, e2e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(A.nbytes + B.nbytes + SA.nbytes + SB.nbytes),
               "d2h_bytes_per_step": int(M * N * out_bytes), "ms_per_step": e2e_ms,
               "schedule": "copy-in / compute / copy-out streams, two buffer sets",
               "steps": n_e2e, "link": link,
               "serial": {"value": job_tflops(flops, ws, serial_ms), "ms_per_step": serial_ms}}

    # ---- further workload shapes (outside the timed region of the headline)
    extras = []
    if not args.no_extra_shapes:
        hbm_gbs, bf16_tf, _, peak_src = load_peaks()
        for label, fname, eM, eN, eK in EXTRA_SHAPES:
            reps = 20 if eM >= 2048 else 100
            cool_down(args)
            us, edesc, ensets = time_shape(mx, dev, fname, eM, eN, eK, reps)
            extras.append(extra_shape_record(label, fname, eM, eN, eK, us, edesc, ensets, hbm_gbs, bf16_tf,
                                             peak_src))

    if rank != 0:
        dist.destroy_process_group()
        return 0

    hbm_gbs, bf16_tf, _, peak_src = load_peaks()
    peak = mx_peak_tflops(fmt_name, bf16_tf)
    gemm_avg_s = statistics.mean(gemm_ms) / 1e3
    achieved = flops / gemm_avg_s / 1e12
    bytes_alg = algorithmic_bytes(M, N, K, fmt_name, out_bytes)
    traffic, traffic_note = read_traffic(fmt_name, M, N, K)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8(e4m3 x e8m0/32) -> f32 accumulate",
        "data": "synthetic",
        "config": {"workload": "mxfp8 NT GEMM M=N=K=4096, E4M3 from N(0,1), E8M0/32, BF16 out",
                   "M": M, "N": N, "K": K, "format": "mxfp8", "out": "bf16",
                   "l2": f"rotating {nsets} input/output sets ({nsets * set_bytes / 2**20:.0f} MiB > 2x L2 "
                         f"{l2 / 2**20:.0f} MiB)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "plan": desc},
        "versions": versions(),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": ("mx_gemm_pair_kernel (CTA-pair tcgen05 block-scaled GEMM)" if "mode=pair" in desc
                                else "mx_gemm_kernel (persistent tcgen05 block-scaled GEMM)"),
                     "peak_source": f"{peak_src} bf16 burst {bf16_tf} TFLOP/s x nominal mxfp8/bf16 ratio "
                                    f"{NOMINAL_PF[fmt_name] / NOMINAL_PF['bf16']:g}",
                     "hbm_view": {"algorithmic_bytes": bytes_alg, "achieved_gbs": bytes_alg / gemm_avg_s / 1e9,
                                  "peak_gbs": hbm_gbs, "frac": bytes_alg / gemm_avg_s / 1e9 / hbm_gbs},
                     "traffic_note": traffic_note},
        "gemm_us": statistics.mean(gemm_ms) * 1e3,
        "gemm_us_event_bracketed": statistics.mean(gemm_bracketed_ms) * 1e3,
        "relayout_us": statistics.mean(relayout_ms) * 1e3,
        "serialised_step_us": serialised_ms * 1e3,
        "wall_ms_per_step": wall_s * 1e3 / args.steps,
        "launch_mode": launch_mode,
        "stream_ms_per_step": stream_total_ms / args.steps,
        "graph_ms_per_step": graph_total_ms / args.steps,
        "gemm_us_stream": gemm_stream_ms * 1e3,
        "gemm_us_graph": gemm_graph_ms * 1e3,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "extra_shapes": extras,
    }
    if not args.no_cpu_baseline:
        rows, dt, threads = oracle_sample_time(A, SA, B, SB, K, fmt, args.cpu_target_s, M)
        line["cpu_baseline"] = {"value": 2.0 * rows * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"rows 0..{rows - 1} of C ({rows}x{N}x{K}), {dt:.1f} s"}
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------- sweep --

def cool_down(args):
    """Idle before timing the next sweep shape: after seconds of a power-capped
    prefill GEMM the GPU keeps its clocks down for a while, and a short kernel
    timed right after measured up to 1.5x slower (MXFP4 8 x 10240 x 8192: 15.5
    us alone, 23.3 us right after 16384 x 57344 x 8192)."""
    if args.sweep_cooldown > 0:
        import torch
        torch.cuda.synchronize()
        time.sleep(args.sweep_cooldown)


def run_sweep(args):
    """Per-shape GEMM time for the model workloads (device-side random codes)."""
    import torch
    from mx_block_scaled_gb300 import binding as mx
    from mx_block_scaled_gb300.inputs import FMT_BY_NAME, WORKLOADS, workload_cases
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, _, peak_src = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    names = args.sweep_workloads.split(",") if args.sweep_workloads else list(WORKLOADS)
    if args.shape:
        M0, N0, K0 = (int(v) for v in args.shape.split(","))
        cases = [("shape", [(args.fmt, 0, 0, M0, N0, K0)])]
    else:
        cases = [(name, list(workload_cases(name))) for name in names]
    for name, wcases in cases:
        seen = set()
        for fmt_name, si, nki, M, N, K in wcases:
            if (fmt_name, M, N, K) in seen:
                continue
            seen.add((fmt_name, M, N, K))
            cool_down(args)
            fmt = FMT_BY_NAME[fmt_name]
            rb = K if fmt_name == "mxfp8" else K // 2
            out = mx.MXGEMM_OUT_BF16 if name == "shape" or WORKLOADS[name]["out"] == "bf16" else mx.MXGEMM_OUT_F32
            ob = 2 if out == mx.MXGEMM_OUT_BF16 else 4
            g = torch.Generator(device=dev)
            g.manual_seed(si * 7919 + nki)

            def codes(rows):
                c = torch.randint(0, 256, (rows, rb), dtype=torch.uint8, device=dev, generator=g)
                if fmt_name == "mxfp8":
                    c = torch.where((c & 0x7F) == 0x7F, c & 0xFE, c)
                return c

            set_bytes = (M + N) * rb + (M + N) * K // 32 + M * N * ob
            nsets = max(2, math.ceil(2 * l2 / set_bytes) + 1)
            nsets = min(nsets, max(2, int(40e9 // set_bytes)))
            plan = mx.Plan(M, N, K, fmt, out, flags=args.sweep_flags, device=dev)
            sets = []
            for _ in range(nsets):
                SA = torch.randint(120, 135, (M, K // 32), dtype=torch.uint8, device=dev, generator=g)
                SB = torch.randint(120, 135, (N, K // 32), dtype=torch.uint8, device=dev, generator=g)
                sets.append((codes(M), mx.relayout_scales(SA, M, K), codes(N), mx.relayout_scales(SB, N, K),
                             torch.empty((M, N), dtype=torch.bfloat16 if ob == 2 else torch.float32, device=dev)))
            # weights are only read: MXGEMM_RUN_B_STATIC lets the decode plans start
            # loading them before the preceding call has finished
            pre = mx.MXGEMM_RUN_SA_PRELAYOUT | mx.MXGEMM_RUN_SB_PRELAYOUT | mx.MXGEMM_RUN_B_STATIC

            def one(i):
                a, sa, b, sb, c = sets[i % nsets]
                st = mx.mxgemm_run(plan.handle, a.data_ptr(), sa.data_ptr(), b.data_ptr(), sb.data_ptr(),
                                   c.data_ptr(), plan.workspace.data_ptr(), plan.ws_bytes, pre,
                                   torch.cuda.current_stream().cuda_stream)
                assert st == 0

            for i in range(3):
                one(i)
            torch.cuda.synchronize()
            reps = args.sweep_reps
            # Replay `reps` calls from a CUDA graph so that host-side launch cost does not
            # show up in the device time of short GEMMs.
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(reps):
                    one(i)
            graph.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) / reps)
            mx.check_device_status()
            del graph
            t = statistics.median(ts) / 1e3
            flops = 2.0 * M * N * K
            byts = algorithmic_bytes(M, N, K, fmt_name, ob)
            peak = mx_peak_tflops(fmt_name, bf16_tf)
            t_roof = max(flops / (peak * 1e12), byts / (hbm_gbs * 1e9))
            print(json.dumps({
                "workload": name, "format": fmt_name, "M": M, "N": N, "K": K, "us": t * 1e6,
                "tflops": flops / t / 1e12, "gbs": byts / t / 1e9,
                "frac_tensor": flops / t / 1e12 / peak, "frac_hbm": byts / t / 1e9 / hbm_gbs,
                "frac_roofline": t_roof / t, "bound": "tensor" if flops / (peak * 1e12) > byts / (hbm_gbs * 1e9)
                else "hbm", "plan": plan.describe(), "nsets": nsets}), flush=True)
            del sets, plan
            torch.cuda.empty_cache()
    return 0


def run_quant_sweep(args):
    """Per-shape time of the MX quantiser (BF16 activations -> codes + tile-layout
    scales) over the activation shapes [M, K] of the model workloads."""
    import torch
    from mx_block_scaled_gb300 import binding as mx
    from mx_block_scaled_gb300.inputs import FMT_BY_NAME, WORKLOADS, workload_cases
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    hbm_gbs, _, _, _ = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    names = args.sweep_workloads.split(",") if args.sweep_workloads else list(WORKLOADS)
    shapes = []
    for name in names:
        for fmt_name, _, _, M, _, K in workload_cases(name):
            if (fmt_name, M, K) not in [(f, m, k) for _, f, m, k in shapes]:
                shapes.append((name, fmt_name, M, K))
    for name, fmt_name, M, K in shapes:
        fmt = FMT_BY_NAME[fmt_name]
        rb = K if fmt_name == "mxfp8" else K // 2
        sf = mx.mxgemm_sf_bytes(M, K)
        byts = M * K * 2 + M * rb + sf
        nsets = max(2, math.ceil(2 * l2 / byts) + 1)
        nsets = min(nsets, max(2, int(20e9 // byts)))
        g = torch.Generator(device=dev)
        g.manual_seed(M * 131 + K)
        sets = [(torch.randn((M, K), dtype=torch.float32, device=dev, generator=g).to(torch.bfloat16),
                 torch.empty((M, rb), dtype=torch.uint8, device=dev),
                 torch.empty(sf, dtype=torch.uint8, device=dev)) for _ in range(nsets)]

        def one(i):
            x, c, t = sets[i % nsets]
            st = mx.mxgemm_quantize(fmt, mx.MXGEMM_IN_BF16, x.data_ptr(), M, K, c.data_ptr(), t.data_ptr(),
                                    mx.MXGEMM_QUANT_SF_TILED, torch.cuda.current_stream().cuda_stream)
            assert st == 0

        for i in range(3):
            one(i)
        torch.cuda.synchronize()
        reps = args.sweep_reps
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(reps):
                one(i)
        graph.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / reps)
        mx.check_device_status()
        del graph
        t = statistics.median(ts) / 1e3
        print(json.dumps({"kernel": "mx_quantize_kernel", "workload": name, "format": fmt_name, "input": "bf16",
                          "M": M, "K": K, "us": t * 1e6, "bytes": byts, "gbs": byts / t / 1e9,
                          "frac_hbm": byts / t / 1e9 / hbm_gbs, "nsets": nsets}), flush=True)
        del sets
        torch.cuda.empty_cache()
    return 0


def run_grouped_sweep(args):
    """Per-case time of the grouped (mixture-of-experts) MX GEMM over the grouped
    workloads: device-side random codes, weight scales laid out once per set,
    token-scale relayout inside each call; CUDA-graph replay over rotating sets."""
    import torch
    from mx_block_scaled_gb300 import binding as mx
    from mx_block_scaled_gb300.inputs import FMT_BY_NAME, MOE_WORKLOADS, group_offsets, moe_cases
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, _, _ = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    names = args.sweep_workloads.split(",") if args.sweep_workloads else list(MOE_WORKLOADS)
    for name in names:
        for fmt_name, nki, G, T, N, K, sizes in moe_cases(name):
            fmt = FMT_BY_NAME[fmt_name]
            rb = K if fmt_name == "mxfp8" else K // 2
            e = 1.0 if fmt_name == "mxfp8" else 0.5
            active = int((sizes > 0).sum())
            flops = 2.0 * float(sizes.sum()) * N * K
            byts = T * K * e + T * K / 32 + active * N * (K * e + K / 32) + T * N * 2
            set_bytes = T * rb + T * K // 32 + G * N * rb + mx.mxgemm_sf_bytes(G * N, K) + T * N * 2
            nsets = max(2, math.ceil(2 * l2 / set_bytes) + 1)
            nsets = min(nsets, max(2, int(30e9 // set_bytes)))
            cool_down(args)
            plan = mx.GroupedPlan(G, T, N, K, fmt, mx.MXGEMM_OUT_BF16, device=dev)
            g = torch.Generator(device=dev)
            g.manual_seed(G * 131 + N + K)

            def codes(rows):
                c = torch.randint(0, 256, (rows, rb), dtype=torch.uint8, device=dev, generator=g)
                if fmt_name == "mxfp8":
                    c = torch.where((c & 0x7F) == 0x7F, c & 0xFE, c)
                return c

            offs = torch.tensor(group_offsets(sizes), dtype=torch.int64, device=dev)
            sets = []
            for _ in range(nsets):
                SB = torch.randint(120, 135, (G * N, K // 32), dtype=torch.uint8, device=dev, generator=g)
                sets.append((codes(T), torch.randint(120, 135, (T, K // 32), dtype=torch.uint8, device=dev,
                                                      generator=g),
                             codes(G * N), mx.relayout_scales(SB, G * N, K),
                             torch.empty((T, N), dtype=torch.bfloat16, device=dev)))
                del SB

            def one(i):
                a, sa, b, sb, c = sets[i % nsets]
                st = mx.mxgemm_grouped_run(plan.handle, offs.data_ptr(), a.data_ptr(), sa.data_ptr(), b.data_ptr(),
                                           sb.data_ptr(), c.data_ptr(), plan.workspace.data_ptr(), plan.ws_bytes,
                                           mx.MXGEMM_RUN_SB_PRELAYOUT, torch.cuda.current_stream().cuda_stream)
                assert st == 0, mx.mxgemm_status_str(st)

            for i in range(3):
                one(i)
            torch.cuda.synchronize()
            reps = args.sweep_reps
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(reps):
                    one(i)
            graph.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) / reps)
            mx.check_device_status()
            del graph
            t = statistics.median(ts) / 1e3
            peak = mx_peak_tflops(fmt_name, bf16_tf)
            t_roof = max(flops / (peak * 1e12), byts / (hbm_gbs * 1e9))
            print(json.dumps({
                "kernel": "mx_gemm_kernel (grouped)", "workload": name, "format": fmt_name, "groups": G,
                "rows": T, "N": N, "K": K, "active_groups": active, "max_group": int(sizes.max()),
                "us": t * 1e6, "tflops": flops / t / 1e12, "gbs": byts / t / 1e9,
                "frac_tensor": flops / t / 1e12 / peak, "frac_hbm": byts / t / 1e9 / hbm_gbs,
                "frac_roofline": t_roof / t,
                "bound": "tensor" if flops / (peak * 1e12) > byts / (hbm_gbs * 1e9) else "hbm",
                "plan": plan.describe(), "nsets": nsets}), flush=True)
            del sets, plan
            torch.cuda.empty_cache()
    return 0


def run_bf16_sweep(args):
    """BF16 NT GEMM (kind::f16 on the same kernels) over the dense workload shapes,
    with cuBLAS (torch.matmul, BF16 in/out) timed the same way as a comparison."""
    import torch
    from mx_block_scaled_gb300 import binding as mx
    from mx_block_scaled_gb300.inputs import WORKLOADS, workload_cases
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    hbm_gbs, bf16_tf, _, _ = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    names = args.sweep_workloads.split(",") if args.sweep_workloads else list(WORKLOADS)
    seen = set()
    shapes = []
    for name in names:
        for _, _, _, M, N, K in workload_cases(name):
            if (M, N, K) not in seen and K % 64 == 0:
                seen.add((M, N, K))
                shapes.append((name, M, N, K))
    for name, M, N, K in shapes:
        byts = (M + N) * K * 2 + M * N * 2
        nsets = max(2, math.ceil(2 * l2 / byts) + 1)
        nsets = min(nsets, max(2, int(30e9 // byts)))
        cool_down(args)
        g = torch.Generator(device=dev)
        g.manual_seed(M + N + K)
        sets = [(torch.randn((M, K), device=dev, generator=g).to(torch.bfloat16),
                 torch.randn((N, K), device=dev, generator=g).to(torch.bfloat16),
                 torch.empty((M, N), dtype=torch.bfloat16, device=dev)) for _ in range(nsets)]
        plan = mx.Plan(M, N, K, mx.MXGEMM_FMT_BF16, mx.MXGEMM_OUT_BF16, device=dev)

        def ours(i):
            a, b, c = sets[i % nsets]
            st = mx.mxgemm_run(plan.handle, a.data_ptr(), 0, b.data_ptr(), 0, c.data_ptr(),
                               plan.workspace.data_ptr(), plan.ws_bytes, 0, torch.cuda.current_stream().cuda_stream)
            assert st == 0, mx.mxgemm_status_str(st)

        def cublas(i):
            a, b, c = sets[i % nsets]
            torch.matmul(a, b.t(), out=c)

        res = {}
        for tag, fn_ in (("ours", ours), ("cublas", cublas)):
            for i in range(3):
                fn_(i)
            torch.cuda.synchronize()
            reps = args.sweep_reps
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(reps):
                    fn_(i)
            graph.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) / reps)
            del graph
            res[tag] = statistics.median(ts) / 1e3
        mx.check_device_status()
        flops = 2.0 * M * N * K
        t_roof = max(flops / (bf16_tf * 1e12), byts / (hbm_gbs * 1e9))
        print(json.dumps({
            "kernel": "mx_gemm (bf16)", "workload": name, "M": M, "N": N, "K": K,
            "us": res["ours"] * 1e6, "tflops": flops / res["ours"] / 1e12,
            "frac_roofline": t_roof / res["ours"],
            "cublas_us": res["cublas"] * 1e6, "cublas_tflops": flops / res["cublas"] / 1e12,
            "cublas_frac_roofline": t_roof / res["cublas"], "speedup_vs_cublas": res["cublas"] / res["ours"],
            "bound": "tensor" if flops / (bf16_tf * 1e12) > byts / (hbm_gbs * 1e9) else "hbm",
            "plan": plan.describe(), "nsets": nsets}), flush=True)
        del sets, plan
        torch.cuda.empty_cache()
    return 0


def run_placement_sweep(args):
    """Scale-placement checker over every pair of valid scale codes (255 x 255) for
    k = 1, 2, 3 elements per operand; prints the time, the tuple rate, the oracle's
    rate on a few pairs, and which pairs agree in both placements."""
    import numpy as np
    import torch
    from mx_block_scaled_gb300 import binding as mx
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    sa, sb = np.meshgrid(np.arange(255, dtype=np.int32), np.arange(255, dtype=np.int32), indexing="ij")
    sa, sb = sa.reshape(-1), sb.reshape(-1)
    dsa, dsb = torch.from_numpy(sa).cuda(), torch.from_numpy(sb).cuda()
    out_dir = args.out_dir  # per-pair counts saved as .npz when given
    for k in (1, 2, 3):
        mx.placement_scan(k, dsa[:64], dsb[:64])  # warm-up
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        counts, first = mx.placement_scan(k, dsa, dsb)
        e1.record(stream)
        torch.cuda.synchronize()
        mx.check_device_status()
        sec = e0.elapsed_time(e1) / 1e3
        c, f = counts.cpu().numpy(), first.cpu().numpy()
        ntup = float(1 << (8 * k)) * len(sa)
        agree = c[:, 0] == 0
        ea, eb = sa.astype(int) - 127, sb.astype(int) - 127
        rec = {"kernel": "placement_scan", "k": k, "pairs": int(len(sa)), "tuples": ntup, "s": sec,
               "tuples_per_s": ntup / sec, "pairs_agreeing": int(agree.sum()),
               "tuples_differing": int(c[:, 0].sum()), "pre_equals_rn": int(c[:, 1].sum()),
               "post_equals_rn": int(c[:, 2].sum())}
        if agree.any():
            rec["agree_ea_range"] = [int(ea[agree].min()), int(ea[agree].max())]
            rec["agree_eb_range"] = [int(eb[agree].min()), int(eb[agree].max())]
            rec["agree_sum_range"] = [int((ea + eb)[agree].min()), int((ea + eb)[agree].max())]
        if out_dir:
            os.makedirs(out_dir, exist_ok=True)
            np.savez_compressed(os.path.join(out_dir, f"placement_k{k}.npz"), sa=sa, sb=sb, counts=c, first=f)
        if not args.no_cpu_baseline and k == 3:
            import oracle
            picks = [(127, 127), (250, 3), (40, 200)]
            t0 = time.perf_counter()
            oracle.placement_scan(k, [p[0] for p in picks], [p[1] for p in picks])
            cpu_s = time.perf_counter() - t0
            rec["cpu_baseline"] = {"kind": "oracle", "tuples_per_s": float(1 << (8 * k)) * len(picks) / cpu_s,
                                   "cores": oracle.num_threads(), "sample": f"{len(picks)} scale pairs at k={k}"}
        print(json.dumps(rec), flush=True)
    return 0


def run_tensor_probe(args):
    """Tensor-pipe rate probe: back-to-back tcgen05.mma from shared-memory operands
    on every SM (or CTA pair), no loads.  One JSON line per (format, cta_group, N,
    scale copies): cycles per MMA, the SM clock the kernel itself saw (clock64 over
    globaltimer: each run lasts milliseconds, too short for nvidia-smi sampling),
    whole-GPU dense PFLOP/s, and that rate against the measured-peak roofline the
    GEMM lines use."""
    import torch
    from mx_block_scaled_gb300 import binding as mx
    torch.cuda.set_device(0)
    _, bf16_tf, _, peak_src = load_peaks()
    fmts = [("mxfp8", mx.MXGEMM_FMT_MXFP8_E4M3), ("mxfp4", mx.MXGEMM_FMT_MXFP4_E2M1), ("bf16", mx.MXGEMM_FMT_BF16)]
    for name, fmt in fmts:
        for cg in (1, 2):
            for n in (128, 256):
                for cp in ((0, 1) if fmt != mx.MXGEMM_FMT_BF16 else (0,)):
                    r = mx.mxgemm_probe_tensor_rate(fmt, cg, n, cp, args.probe_stages)
                    peak = mx_peak_tflops(name, bf16_tf) / 1e3
                    rec = {"kernel": "tensor_rate_probe", "fmt": name, "cta_group": cg, "n": n,
                           "scale_copies": bool(cp), "stages": args.probe_stages,
                           "m_per_mma": 128 * cg, "cycles_per_mma": round(r["cycles_per_mma"], 2),
                           "sm_ghz": round(r["sm_ghz"], 3), "units": r["units"], "pflops": round(r["pflops"], 3),
                           "peak_pflops": round(peak, 3), "frac_of_peak": round(r["pflops"] / peak, 3),
                           "peak_src": f"{peak_src} bf16 x nominal {name}/bf16"}
                    print(json.dumps(rec), flush=True)
    return 0


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def run_oracle_sweep(args):
    """The CPU oracle (the baseline, not a target) on the host cores: the full
    product for the 256^3 and 4096^3 cases and every shape with M <= 256, the
    first rows of C extrapolated linearly for larger M (labelled), and a
    single-core rate on 4096^3.  Operand values do not change the oracle's
    speed; seeded finite random codes stand in for the workloads' values."""
    import numpy as np
    import oracle
    from mx_block_scaled_gb300.inputs import FMT_BY_NAME, WORKLOADS, finite_uniform_codes, workload_cases
    threads = oracle.num_threads()
    print(json.dumps({"kind": "oracle", "cpu": _cpu_model(), "threads": threads}), flush=True)
    seen = set()
    for name in WORKLOADS:
        for fmt_name, si, nki, M, N, K in workload_cases(name):
            if (fmt_name, M, N, K) in seen:
                continue
            seen.add((fmt_name, M, N, K))
            fmt = FMT_BY_NAME[fmt_name]
            rng = np.random.default_rng([M, N, K, fmt])
            full = M <= 256 or (M, N, K) == (4096, 4096, 4096)
            rows = M if full else min(M, 64)
            A, SA = finite_uniform_codes(rng, rows, K, fmt, 120, 134)
            B, SB = finite_uniform_codes(rng, N, K, fmt, 120, 134)
            t0 = time.perf_counter()
            oracle.gemm(fmt, A, SA, B, SB, K, with_abs=False)
            dt = time.perf_counter() - t0
            sec = dt * (M / rows)
            print(json.dumps({"kind": "oracle", "workload": name, "format": fmt_name, "M": M, "N": N, "K": K,
                              "seconds": sec, "mode": "full" if full else f"extrapolated from {rows} rows",
                              "threads": threads, "tflops": 2.0 * M * N * K / sec / 1e12}), flush=True)
    # one core, 4096^3 (first 64 rows, extrapolated)
    rng = np.random.default_rng(1)
    A, SA = finite_uniform_codes(rng, 64, 4096, FMT_BY_NAME["mxfp8"], 120, 134)
    B, SB = finite_uniform_codes(rng, 4096, 4096, FMT_BY_NAME["mxfp8"], 120, 134)
    t0 = time.perf_counter()
    oracle.gemm(FMT_BY_NAME["mxfp8"], A, SA, B, SB, 4096, with_abs=False, nthreads=1)
    dt = time.perf_counter() - t0
    print(json.dumps({"kind": "oracle", "workload": "mxfp8_square_4096", "format": "mxfp8", "M": 4096, "N": 4096,
                      "K": 4096, "seconds": dt * 64, "mode": "extrapolated from 64 rows", "threads": 1,
                      "tflops": 2.0 * 4096 ** 3 / (dt * 64) / 1e12}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--soak-s", type=float, default=2.0, help="untimed load before the timed region (clocks)")
    ap.add_argument("--cpu-target-s", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra-shapes", action="store_true",
                    help="skip the further workload shapes timed after the headline")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-workloads", default="")
    ap.add_argument("--sweep-reps", type=int, default=20)
    ap.add_argument("--sweep-flags", type=int, default=0, help="mxgemm_plan_create flags for --sweep")
    ap.add_argument("--sweep-cooldown", type=float, default=3.0,
                    help="seconds of idle before each sweep shape (lets the clocks recover from the last one)")
    ap.add_argument("--shape", default="", help="M,N,K: sweep this one shape (BF16 out)")
    ap.add_argument("--fmt", default="mxfp8", choices=["mxfp8", "mxfp4"], help="format for --shape")
    ap.add_argument("--quant-sweep", action="store_true",
                    help="time the MX quantiser over the workloads' activation shapes")
    ap.add_argument("--bf16-sweep", action="store_true",
                    help="time the BF16 NT GEMM (and cuBLAS beside it) over the dense workload shapes")
    ap.add_argument("--grouped-sweep", action="store_true",
                    help="time the grouped (mixture-of-experts) MX GEMM over the grouped workloads")
    ap.add_argument("--oracle-sweep", action="store_true",
                    help="time the CPU oracle over the workload shapes (full for M <= 256, else extrapolated)")
    ap.add_argument("--out-dir", default="", help="--placement-sweep: save the per-pair counts here (.npz)")
    ap.add_argument("--placement-sweep", action="store_true",
                    help="run the scale-placement checker over every scale pair for k = 1, 2, 3")
    ap.add_argument("--tensor-probe", action="store_true",
                    help="measure the tensor pipe's own MMA rate (operands resident in shared memory)")
    ap.add_argument("--probe-stages", type=int, default=16384, help="k-stages per unit for --tensor-probe")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.quant_sweep:
        return run_quant_sweep(args)
    if args.grouped_sweep:
        return run_grouped_sweep(args)
    if args.bf16_sweep:
        return run_bf16_sweep(args)
    if args.placement_sweep:
        return run_placement_sweep(args)
    if args.oracle_sweep:
        return run_oracle_sweep(args)
    if args.tensor_probe:
        return run_tensor_probe(args)
    if args.sweep or args.shape:
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
