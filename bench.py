#!/usr/bin/env python
"""Benchmark of the MXFP4 routed expert linear on one GB300 (or N replicas).

One step = one call of the whole path (routing bucketer, routed expert
linear, combine) over one batch of a named workload, inputs resident in HBM.
The headline workload is the largest single-GPU one, skewed prefill (T=8192
tokens, E=384 experts, K=8 picks from Zipf(1.2) popularity, I=7168,
O=4096, bf16 tokens, MXFP4 weights); decode, wide decode and prefill are
measured in the same run and reported under "configs", each with its own
roofline, end-to-end number, clocks and CPU baseline. Seeded synthetic data.

Prints one JSON line (rank 0). The path does not exchange data between
GPUs: with --gpus N every rank runs its own replica (weak scaling) and the
value is the work all ranks did divided by the slowest rank's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--configs all|none|a,b]
  python bench.py --impl reference ...   # the float64 CPU oracle, timed
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed-expert GB/s and TFLOP/s at 1 GB300, % of HBM/bf16 roofline"
FLUSH_BYTES = 512 << 20          # > 129 MB of L2: written between steps
# The headline: the largest single-GPU workload (8192 tokens, 384 experts,
# 8 picks, Zipf(1.2) popularity); the others are measured in the same run.
HEADLINE = "skewed_prefill"
ALL_CONFIGS = ("decode", "wide_decode", "prefill", "skewed_prefill")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    help="the workload of the line's headline value")
    ap.add_argument("--configs", default="all",
                    help="other workloads measured in the same run and reported under "
                         "'configs': 'all', 'none' or a comma-separated list")
    ap.add_argument("--weights", choices=["plain", "prepared"], default="plain",
                    help="weights as given (plain) or laid out once for the kernels before "
                         "timing (prepared: mxfp4_expert_linear_prepare, load-time work)")
    ap.add_argument("--no-prepared-leg", action="store_true",
                    help="with plain weights, skip the extra timing on prepared weights")
    ap.add_argument("--cpu-budget", type=float, default=6.0,
                    help="seconds of oracle time per workload for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the router and SwiGLU-expert fields (clean launch lists)")
    ap.add_argument("--swiglu-only", action="store_true",
                    help="time only the SwiGLU expert at the workload's layer shape")
    return ap.parse_args()


# ----------------------------------------------------------- accounting ----
def token_bytes(wl):
    import torch
    return 2 if wl.dtype == torch.bfloat16 else 4


def per_expert_bytes(wl):
    G = wl.I // 32
    return wl.O * G * 16 + wl.O * G           # packed bytes + scale bytes


def path_bytes(wl, U, T=None):
    """Algorithmic bytes of the whole path: selected experts' packed bytes and
    scales, tokens, shared output read, output written, routing (sel + p)."""
    T = wl.T if T is None else T
    bx = token_bytes(wl)
    return U * per_expert_bytes(wl) + T * wl.I * bx + 2 * T * wl.O * bx + T * wl.K * 8


def linear_bytes(wl, U):
    """Algorithmic bytes of the routed linear kernel: selected weights + tokens."""
    return U * per_expert_bytes(wl) + wl.T * wl.I * token_bytes(wl)


def path_flops(wl, T=None):
    T = wl.T if T is None else T
    return 2 * T * wl.K * wl.O * wl.I


def workload_is_hbm_bound(wl, U, peaks):
    return (path_bytes(wl, U) / (peaks["hbm_gbs"] * 1e9)
            >= path_flops(wl) / (peaks["bf16_tflops"] * 1e12))


def sample_metric(wl, rows, hbm_bound, seconds):
    """The metric for a token sample of the workload computed in `seconds`."""
    if hbm_bound:
        return sample_bytes(wl, rows) / seconds / 1e9, "GB/s"
    return path_flops(wl, T=len(rows)) / seconds / 1e12, "TFLOP/s"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


KERNEL_SOURCES = {
    "gemv_kernel": ["mxfp4_routed_expert_route_gb300/csrc/gemv.cu",
                    "mxfp4_routed_expert_route_gb300/csrc/common.cuh",
                    "mxfp4_routed_expert_route_gb300/csrc/internal.h",
                    "mxfp4_routed_expert_route_gb300/csrc/prepare.cu"],
    "gemm_tc_kernel": ["mxfp4_routed_expert_route_gb300/csrc/gemm_tc.cu",
                       "mxfp4_routed_expert_route_gb300/csrc/common.cuh",
                       "mxfp4_routed_expert_route_gb300/csrc/internal.h",
                       "mxfp4_routed_expert_route_gb300/csrc/prepare.cu"],
}


def ncu_traffic(kernel, workload, layout="plain"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source, this workload and this weight layout; else
    None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    key = f"{kernel}/{workload}" + ("/prepared" if layout == "prepared" else "")
    try:
        with open(path) as f:
            d = json.load(f)[key]
    except (OSError, ValueError, KeyError):
        return None
    if d.get("source_sha256") != source_digest(KERNEL_SOURCES[kernel]):
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------- across ranks ----
def max_over_ranks(seconds, device, world):
    """The slowest rank's time: every rank passes its own and gets the max
    (all-reduce MAX on `device`, which is the GPU for NCCL and the CPU for
    gloo)."""
    import torch
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step, steps, world, t_max_s):
    """Units all ranks processed per second: every rank runs the same
    replica (weak scaling), timed by the slowest rank."""
    return world * units_per_rank_step * steps / t_max_s


# --------------------------------------------------------------- clocks ----
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str, interval_ms: int = 20):
        self.cmd = ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", "-lms", str(interval_ms)]
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)              # let the first sample land before the load

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(device_index):
    import torch
    props = torch.cuda.get_device_properties(device_index)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        s = str(uuid)
        return s if s.startswith("GPU-") else "GPU-" + s
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    return vis.split(",")[device_index] if vis else str(device_index)


# -------------------------------------------------------------- oracle -----
def oracle_sample_time(wl, rows):
    import oracle
    t0 = time.perf_counter()
    oracle.expert_linear(wl.x, wl.packed, wl.scales, wl.sel, wl.p, wl.y_shared,
                         rows=rows)
    return time.perf_counter() - t0


def sample_bytes(wl, rows):
    import numpy as np
    sel = wl.sel.numpy()[rows]
    U = len(np.unique(sel[(sel >= 0) & (sel < wl.E)]))
    return path_bytes(wl, U, T=len(rows))


def cpu_baseline(wl, hbm_bound, budget_s=6.0):
    """The oracle as it stands on this host's cores, on a bounded token sample."""
    import numpy as np
    import oracle
    one = oracle_sample_time(wl, np.array([0]))
    n = int(max(1, min(wl.T, budget_s / max(one, 1e-6))))
    rows = np.arange(n)
    t = oracle_sample_time(wl, rows)
    v, unit = sample_metric(wl, rows, hbm_bound, t)
    return {"value": v, "unit": unit,
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"tokens 0..{n - 1} of the {wl.name} batch ({n}/{wl.T}), "
                      f"all O={wl.O} rows, one run of {t:.2f} s"}


def workload_config(wl, U, world):
    """The workload description both arms print as ``config``."""
    return {"workload": wl.name, "T": wl.T, "E": wl.E, "K": wl.K, "I": wl.I, "O": wl.O,
            "tokens": "bf16" if token_bytes(wl) == 2 else "fp32",
            "weights": "mxfp4 (e2m1 codes + e8m0 scale per 32)",
            "picks": wl.meta["picks"], "experts_touched": U, "seed": wl.meta["seed"],
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank):
    """Reference arm: the float64 CPU oracle, timed as it stands."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from mxfp4_routed_expert_route_gb300 import workloads
    oracle.build()
    wl = workloads.named(args.workload)
    one = oracle_sample_time(wl, np.array([0]))
    budget = 120.0
    n = int(max(1, min(wl.T, budget / max(one * (args.steps + args.warmup), 1e-9))))
    rows = np.arange(n)
    for _ in range(args.warmup):
        oracle_sample_time(wl, rows)
    times = [oracle_sample_time(wl, rows) for _ in range(args.steps)]
    mean = sum(times) / len(times)
    peaks, _ = load_peaks()
    U = workloads.experts_touched(wl.sel, wl.E)
    value, unit = sample_metric(wl, rows, workload_is_hbm_bound(wl, U, peaks), mean)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, U, 1),
        "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"tokens 0..{n - 1} of the {wl.name} batch "
                                   f"({n}/{wl.T}), all O={wl.O} rows, per step"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ours -----
def measure_router(wl, d, dev, stream, flush, warmup, n, peaks):
    """The router that feeds the linear (sigmoid top-K from logits, seeded
    N(0,1) float32 logits, zero bias so that the routing is as balanced as
    the workload's own picks): alone, and fused with the linear in one
    library call; CUDA events on the stream, L2 flushed before each call,
    medians."""
    import torch
    from mxfp4_routed_expert_route_gb300 import mxfp4_expert_linear_routed, router_topk
    g = torch.Generator().manual_seed(1000 + wl.meta["seed"])
    lg = torch.randn(wl.T, wl.E, generator=g).to(dev)
    bias = torch.zeros(wl.E, device=dev)
    out = torch.empty((wl.T, wl.O), dtype=wl.dtype, device=dev)

    def routed():
        mxfp4_expert_linear_routed(d["x"], d["packed"], d["scales"], lg, bias, wl.K,
                                   d["y_shared"], out=out)

    def timed(fn):
        for _ in range(warmup):
            flush.zero_()
            fn()
        ev = []
        for _ in range(n):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize(dev)
        ts = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
        return ts[len(ts) // 2]

    us = timed(lambda: router_topk(lg, bias, wl.K))
    routed_us = timed(routed)
    nbytes = wl.T * wl.E * 4 + wl.E * 4 + wl.T * wl.K * 8
    gbps = nbytes / (us * 1e-6) / 1e9
    return {"us": us, "bytes": nbytes, "gbps": gbps, "frac_of_hbm": gbps / peaks["hbm_gbs"],
            "routed_call_us": routed_us,
            "inputs": "seeded N(0,1) float32 logits, zero bias, scaling 1"}


SWIGLU_FOR = {"decode": "swiglu_decode", "prefill": "swiglu_prefill"}
ROUTER_FOR = ("decode", "prefill")


def measure_swiglu(name, dev, stream, flush, warmup, n, peaks):
    """The whole routed SwiGLU expert (gate/up linear, SwiGLU, down linear,
    combine) at the layer shape of the named workload: one library call, CUDA
    events on the stream, L2 flushed before each call, median. Its roofline
    is the slower of the algorithmic bytes (selected experts' gate/up and
    down bytes and scales, tokens, shared output, output, routing) at HBM
    bandwidth and its FLOPs at the bf16 peak."""
    import torch
    from mxfp4_routed_expert_route_gb300 import (mxfp4_swiglu_expert, swiglu_workspace_size,
                                                 workloads)
    wl = workloads.named_swiglu(name)
    d = wl.device_tensors(dev)
    out = torch.empty((wl.T, wl.O), dtype=wl.dtype, device=dev)
    ws = torch.empty(max(1, swiglu_workspace_size(wl.T, wl.E, wl.I, wl.F, wl.O, wl.K,
                                                  wl.dtype)), dtype=torch.uint8, device=dev)

    def call():
        mxfp4_swiglu_expert(*[d[k] for k in wl.ARGS], out=out, workspace=ws)

    for _ in range(warmup):
        flush.zero_()
        call()
    ev = []
    for _ in range(n):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize(dev)
    ts = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
    us = ts[len(ts) // 2]
    U = workloads.experts_touched(wl.sel, wl.E)
    bx = token_bytes(wl)
    per_expert = 2 * wl.F * (wl.I // 32) * 17 + wl.O * (wl.F // 32) * 17
    nbytes = (U * per_expert + wl.T * wl.I * bx + 2 * wl.T * wl.O * bx + wl.T * wl.K * 8)
    flops = 2 * wl.T * wl.K * (2 * wl.F * wl.I + wl.O * wl.F)
    t_roof = max(nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    hbm = nbytes / (peaks["hbm_gbs"] * 1e9) >= flops / (peaks["bf16_tflops"] * 1e12)
    return {"workload": name, "T": wl.T, "E": wl.E, "K": wl.K, "I": wl.I, "F": wl.F,
            "O": wl.O, "experts_touched": U, "us": us, "bytes_alg": nbytes, "flops_alg": flops,
            "gbps": nbytes / (us * 1e-6) / 1e9, "tflops": flops / (us * 1e-6) / 1e12,
            "bound": "hbm" if hbm else "tensor", "t_roof_us": t_roof * 1e6,
            "frac": t_roof / (us * 1e-6)}


def f16_tile_share(wl, rows_per_tile=128, max_span=26):
    """Share of the tensor-core kernel's 128-row weight tiles that run on f16
    operands: those whose every row's scale bytes span at most 26 binades
    (the others run on bf16)."""
    import numpy as np

    sc = wl.scales.numpy()
    span = sc.max(axis=-1).astype(np.int16) - sc.min(axis=-1).astype(np.int16)   # (E, O)
    E, O = span.shape
    tiles = -(-O // rows_per_tile)
    pad = np.zeros((E, tiles * rows_per_tile), dtype=np.int16)
    pad[:, :O] = span
    ok = (pad.reshape(E, tiles, rows_per_tile) <= max_span).all(axis=-1)
    return float(ok.mean())


def linear_dtype_label(wl, gemm):
    """What the routed linear computes in, for the line's ``dtype``."""
    if gemm:
        share = f16_tile_share(wl)
        return (f"f16 x f16 -> f32 on {100 * share:.0f}% of weight tiles, bf16 x bf16 -> f32 on "
                "the rest (tensor cores; MXFP4 decoded exactly, with powers of two per weight "
                "row and per token)")
    if token_bytes(wl) == 2:
        return "f16x2 products summed in chains of 8, f32 across groups (bf16 tokens)"
    return "f32"


def measure_prepared(wl, d, dev, stream, flush, W, K, lib, world, gemm, bytes_step,
                     flops_step, t_roof, hbm_bound, plain_roofline):
    """The same steps on weights laid out once by mxfp4_expert_linear_prepare
    (load-time work, before timing): whole-step time (L2 flushed between
    steps) and the routed-linear kernel's CUDA-event time."""
    import ctypes

    import torch

    from mxfp4_routed_expert_route_gb300 import (_native, mxfp4_expert_linear_prepared,
                                                 prepare_weights, prepared_workspace_size)

    pw = prepare_weights(d["packed"], d["scales"])
    ws = torch.empty(max(1, prepared_workspace_size(wl.T, wl.E, wl.I, wl.O, wl.K, wl.dtype)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((wl.T, wl.O), dtype=wl.dtype, device=dev)

    def step():
        mxfp4_expert_linear_prepared(d["x"], pw, d["sel"], d["p"], d["y_shared"], out=out,
                                     workspace=ws)

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e

    for _ in range(W):
        flush.zero_()
        step()
    steps = [(ev(), ev()) for _ in range(K)]
    lin = [(ev(), ev()) for _ in range(K)]
    torch.cuda.synchronize(dev)
    for i in range(K):
        flush.zero_()
        steps[i][0].record(stream)
        step()
        steps[i][1].record(stream)
    torch.cuda.synchronize(dev)
    for i in range(K):
        flush.zero_()
        lib.mxfp4el_set_stage_events(_native.STAGE_LINEAR, ctypes.c_void_p(lin[i][0].cuda_event),
                                     ctypes.c_void_p(lin[i][1].cuda_event))
        step()
    torch.cuda.synchronize(dev)
    lib.mxfp4el_set_stage_events(_native.STAGE_LINEAR, None, None)
    t = max_over_ranks(sum(a.elapsed_time(b) for a, b in steps) / 1e3, dev, world)
    lin_s = sum(a.elapsed_time(b) for a, b in lin) / K / 1e3
    rate = whole_job_rate(bytes_step if hbm_bound else flops_step, K, world, t)
    units = plain_roofline.get("flops_per_launch") or plain_roofline.get("bytes_per_launch")
    achieved = units / lin_s / (1e12 if gemm else 1e9)
    return {"weights_layout": "prepared once before timing (mxfp4_expert_linear_prepare)",
            "value": rate / (1e9 if hbm_bound else 1e12), "ms_per_step": t / K * 1e3,
            "path_roofline_frac": t_roof / (t / K),
            "kernel": {"launch_us": lin_s * 1e6, "achieved": achieved,
                       "unit": plain_roofline["unit"],
                       "frac": achieved / plain_roofline["peak"],
                       "traffic": ncu_traffic("gemm_tc_kernel" if gemm else "gemv_kernel",
                                              wl.name, "prepared")}}


def measure_workload(name, args, lib, dev, rank, world):
    """Every number of one workload: whole steps (device-timed, L2 flushed),
    the dominant kernel's CUDA-event duration inside the same steps, the
    end-to-end steps through the public call with pinned host I/O, the
    router and SwiGLU extras where they apply, and the oracle's CPU
    baseline (rank 0 at N=1)."""
    import ctypes

    import torch
    import torch.distributed as dist

    from mxfp4_routed_expert_route_gb300 import (_native, mxfp4_expert_linear,
                                                 mxfp4_expert_linear_prepared, prepare_weights,
                                                 prepared_workspace_size, workloads,
                                                 workspace_size)

    wl = workloads.named(name)
    U = workloads.experts_touched(wl.sel, wl.E)
    d = wl.device_tensors(dev)
    out = torch.empty((wl.T, wl.O), dtype=wl.dtype, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    if args.weights == "prepared":
        # Load-time work, before any timing: the weights laid out for the
        # kernels once; every step then reads the prepared copy.
        pw = prepare_weights(d["packed"], d["scales"])
        ws = torch.empty(max(1, prepared_workspace_size(wl.T, wl.E, wl.I, wl.O, wl.K,
                                                        wl.dtype)),
                         dtype=torch.uint8, device=dev)

        def call(x, sel, p, ys, o):
            mxfp4_expert_linear_prepared(x, pw, sel, p, ys, out=o, workspace=ws)
    else:
        ws = torch.empty(max(1, workspace_size(wl.T, wl.E, wl.I, wl.O, wl.K, wl.dtype)),
                         dtype=torch.uint8, device=dev)

        def call(x, sel, p, ys, o):
            mxfp4_expert_linear(x, d["packed"], d["scales"], sel, p, ys, out=o, workspace=ws)

    def step():
        call(d["x"], d["sel"], d["p"], d["y_shared"], out)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()

    def new_event():
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(stream)                 # creates the underlying CUDA event
        return ev

    K, W = args.steps, args.warmup
    for _ in range(W):
        flush.zero_()
        step()

    # Timed loop A: whole steps, for the value. Nothing is recorded between
    # the library's kernels, so their launches may overlap.
    ev = [(new_event(), new_event()) for _ in range(K)]
    barrier()
    sampler = ClockSampler(gpu_id_for(dev.index))
    sampler.start()
    launches0 = lib.mxfp4el_kernel_launches()
    barrier()
    t0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    barrier()
    wall = time.perf_counter() - t0
    launches = lib.mxfp4el_kernel_launches() - launches0
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # Timed loop B: the same steps with CUDA events around the routed-linear
    # kernel's launch (on the library's stream), for its roofline fraction.
    lin = [(new_event(), new_event()) for _ in range(K)]
    barrier()
    for i in range(K):
        flush.zero_()
        lib.mxfp4el_set_stage_events(_native.STAGE_LINEAR,
                                     ctypes.c_void_p(lin[i][0].cuda_event),
                                     ctypes.c_void_p(lin[i][1].cuda_event))
        step()
    barrier()
    lib.mxfp4el_set_stage_events(_native.STAGE_LINEAR, None, None)
    lin_ms = [a.elapsed_time(b) for a, b in lin]

    t_max = max_over_ranks(sum(step_ms) / 1e3, dev, world)

    # End to end through the public API: pinned host inputs in, result out,
    # every step's copies inside the timed span. The steps are pipelined: the
    # inputs of step i+1 are copied on a copy stream while step i computes,
    # and step i's result is read back on a third stream (device inputs and
    # outputs double-buffered, ordered by events). No L2 flush here: every
    # step streams more than L2 holds (its selected weights alone).
    # The step's inputs (tokens, ids, weights, shared output) packed into one
    # pinned buffer, 256-byte aligned pieces, so that one copy moves them.
    host_in = (wl.x, wl.sel, wl.p, wl.y_shared)
    sizes = [t.numel() * t.element_size() for t in host_in]
    offs, total = [], 0
    for n in sizes:
        offs.append(total)
        total += (n + 255) // 256 * 256
    pack_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(host_in, offs, sizes):
        pack_h[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))

    def views(buf):
        return [buf[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(host_in, offs, sizes)]

    out_h = [torch.empty((wl.T, wl.O), dtype=wl.dtype).pin_memory() for _ in range(2)]
    pack_d = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    bufs = [views(pack_d[b]) + [torch.empty((wl.T, wl.O), dtype=wl.dtype, device=dev)]
            for b in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # Per buffer slot: inputs landed, step computed, result read back.
    h2d_ev, comp_ev, d2h_ev = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def e2e_run(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_h2d)
        for i in range(n):
            b = i % 2
            x_d, sel_d, p_d, ys_d, out_d = bufs[b]
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(comp_ev[b])            # step i-2 has read this buffer
                pack_d[b].copy_(pack_h, non_blocking=True)
                h2d_ev[b].record(s_h2d)
            stream.wait_event(h2d_ev[b])
            if i >= 2:
                stream.wait_event(d2h_ev[b])                # step i-2's result is read back
            call(x_d, sel_d, p_d, ys_d, out_d)
            comp_ev[b].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(comp_ev[b])
                out_h[b].copy_(out_d, non_blocking=True)
                d2h_ev[b].record(s_d2h)
        end.record(s_d2h)                                  # after the last read-back
        return start, end

    e2e_run(W)
    barrier()
    e2e_start, e2e_end = e2e_run(K)
    barrier()
    e2e_max = max_over_ranks(e2e_start.elapsed_time(e2e_end) / 1e3, dev, world)
    h2d = sum(sizes)
    d2h = out_h[0].numel() * out_h[0].element_size()

    peaks, peaks_src = load_peaks()
    extras = not args.no_extras
    router = (measure_router(wl, d, dev, stream, flush, W, min(K, 200), peaks)
              if extras and wl.name in ROUTER_FOR else None)
    swiglu = (measure_swiglu(SWIGLU_FOR[wl.name], dev, stream, flush, W, min(K, 100), peaks)
              if extras and wl.name in SWIGLU_FOR else None)
    gemm = lib.mxfp4el_linear_path(wl.T, wl.E, wl.I, wl.O, wl.K,
                                   _native.DTYPE_BF16 if token_bytes(wl) == 2
                                   else _native.DTYPE_F32) == _native.PATH_GEMM
    bytes_step = path_bytes(wl, U)
    flops_step = path_flops(wl)
    t_roof = max(bytes_step / (peaks["hbm_gbs"] * 1e9),
                 flops_step / (peaks["bf16_tflops"] * 1e12))
    hbm_bound = workload_is_hbm_bound(wl, U, peaks)
    gbps = whole_job_rate(bytes_step, K, world, t_max) / 1e9
    tflops = whole_job_rate(flops_step, K, world, t_max) / 1e12
    value, unit = (gbps, "GB/s") if hbm_bound else (tflops, "TFLOP/s")
    ms_step = t_max / K * 1e3
    lin_mean_s = sum(lin_ms) / len(lin_ms) / 1e3
    if gemm:
        kernel = "gemm_tc_kernel"
        lin_flops = 2.0 * int((wl.sel >= 0).sum()) * wl.O * wl.I
        achieved = lin_flops / lin_mean_s / 1e12
        peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        roofline = {"bound": "tensor", "kernel": "gemm_tc_kernel (routed expert grouped GEMM)",
                    "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak,
                    "peak_source": f"bf16_tflops_sustained of {peaks_src} "
                                   f"(burst {peaks['bf16_tflops']}: "
                                   f"frac {achieved / peaks['bf16_tflops']:.3f})",
                    "flops_per_launch": lin_flops, "launch_us": lin_mean_s * 1e6}
    else:
        kernel = "gemv_kernel"
        lin_bytes = linear_bytes(wl, U)
        achieved = lin_bytes / lin_mean_s / 1e9
        roofline = {"bound": "hbm", "kernel": "gemv_stream_kernel (routed expert linear)",
                    "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"],
                    "peak_source": f"hbm_gbs of {peaks_src}",
                    "bytes_per_launch": lin_bytes, "launch_us": lin_mean_s * 1e6}
    roofline["traffic"] = ncu_traffic(kernel, wl.name, args.weights)
    e2e_v = whole_job_rate(bytes_step if hbm_bound else flops_step, K, world, e2e_max)
    res = {
        "value": value, "unit": unit, "ms_per_step": ms_step,
        "dtype": linear_dtype_label(wl, gemm),
        "config": workload_config(wl, U, world),
        "weights_layout": ("prepared once before timing (mxfp4_expert_linear_prepare, "
                           "load-time work)" if args.weights == "prepared"
                           else "plain layout as given"),
        "linear": "tensor-core grouped GEMM" if gemm else "CUDA-core GEMV",
        "l2": f"flushed between steps ({FLUSH_BYTES >> 20} MiB write)",
        "gbps": gbps, "tflops": tflops,
        "path_roofline": {"t_roof_us": t_roof * 1e6, "t_step_us": ms_step * 1e3,
                          "frac": t_roof / (ms_step / 1e3), "bytes_alg": bytes_step,
                          "flops_alg": flops_step, "peaks": peaks_src,
                          "bound": "hbm" if hbm_bound else "tensor"},
        "roofline": roofline,
        "e2e": {"value": e2e_v / (1e9 if hbm_bound else 1e12), "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_max / K * 1e3,
                "schedule": "steps pipelined: step i+1's inputs copied while step i "
                            "computes, double-buffered; all copies inside the timed span",
                "l2": "not flushed: each step streams more than L2 (its selected weights)"},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "wall_s": wall,
    }
    if args.weights == "plain" and not args.no_prepared_leg:
        res["prepared"] = measure_prepared(wl, d, dev, stream, flush, W, K, lib, world, gemm,
                                           bytes_step, flops_step, t_roof, hbm_bound, roofline)
    if router is not None:
        res["router"] = router
    if swiglu is not None:
        res["swiglu_expert"] = swiglu
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, hbm_bound, budget_s=args.cpu_budget)
    return res


def run_ours(args, rank, world):
    import torch

    from mxfp4_routed_expert_route_gb300 import _native, build

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    lib = _native.load()

    names = [args.workload]
    if args.configs != "none":
        listed = ALL_CONFIGS if args.configs == "all" else args.configs.split(",")
        names = [n for n in listed if n != args.workload] + [args.workload]
    results = {}
    for name in names:
        results[name] = measure_workload(name, args, lib, dev, rank, world)
        torch.cuda.empty_cache()
    if rank != 0:
        return
    head = results[args.workload]
    line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": head["dtype"], "data": "synthetic"}
    line.update({k: v for k, v in head.items() if k not in line and k != "value"})
    if len(results) > 1:
        line["configs"] = {n: results[n] for n in ALL_CONFIGS if n in results}
        line["configs"].update({n: r for n, r in results.items() if n not in line["configs"]})
    print(json.dumps(line), flush=True)


def run_swiglu_only(args, rank):
    """The SwiGLU expert alone at the workload's layer shape (for profiling)."""
    import torch
    from mxfp4_routed_expert_route_gb300 import build
    if args.workload not in SWIGLU_FOR:
        raise SystemExit(f"no SwiGLU shape for workload {args.workload}")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    peaks, _ = load_peaks()
    r = measure_swiglu(SWIGLU_FOR[args.workload], dev, torch.cuda.current_stream(dev), flush,
                       args.warmup, args.steps, peaks)
    if rank == 0:
        print(json.dumps(r), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        if args.swiglu_only:
            run_swiglu_only(args, rank)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
