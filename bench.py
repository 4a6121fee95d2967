#!/usr/bin/env python3
"""Throughput of the blockwise-FP8 routed-MoE layer on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl native|reference]

A step is one pass of the whole layer (router, permutation, gate/up + SwiGLU,
down, combine) over one synthetic batch already resident in HBM.  The L2 is
flushed before every step (a 256 MiB memset, twice the 129 MB L2, then a
read of another 256 MiB so that no dirty line of the memset is left to be
written back inside the timed step) and the step is timed with CUDA events
on the launching stream.  The default workload is the largest single-GPU
configuration, the large prefill batch (T=4096, H=6144, E=512, top-12,
I=2048, router bias N(0, 1)); ``--workload`` selects the others (e.g.
olmoe_decode_T8, olmoe_prefill_T2048, wide_decode_T64).

Printed: ONE JSON line.  Besides the contract keys it carries
  roofline      : the dominant kernel's algorithmic bytes (or FLOPs) per launch
                  over its CUDA-event duration, against MEASURED_PEAKS.json
                  (the gate/up GEMM on prefill batches also gives its FP8
                  TFLOP/s and the attainable fraction max(bytes / bandwidth,
                  FLOPs / FP8 peak) / time);
  layer         : the same for the whole step (selected-expert bytes / step);
  cpu_baseline  : the f64 CPU oracle, threaded over tokens (router) and expert
                  segments (FFN) on all host cores, on a bounded sample;
  e2e           : the metric through the host-buffer C-ABI entry point;
  kernels_us    : per-kernel-step CUDA-event times from a few extra steps
                  after the timed region (events between the kernels);
  clocks        : nvidia-smi samples taken during the timed region.
``--impl reference`` times the CPU oracle as the reference arm instead.
Under torchrun (N > 1) every rank runs an independent replica.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "MoE-layer tokens/s; decode HBM GB/s & prefill FP8 TFLOP/s vs roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "large_prefill_T4096"
# the library's timed kernel steps (a step may be two chained kernels)
KERNEL_STEPS = ("route", "router_logits", "router_select", "permute", "act_quant", "gate_up",
                "down", "combine")
FLUSH_BYTES = 256 << 20
FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor throughput on GB300 (4.5 / 2.25 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "gemv", "gemm", "tcgemv"],
                    help="force one of the layer's expert paths (default: the library's choice)")
    ap.add_argument("--format", default="fp8", choices=["fp8", "nvfp4"],
                    help="expert weight format: blockwise e4m3 (default) or NVFP4 (e2m1 + e4m3 "
                         "scale per 16 weights + f32 global per expert matrix)")
    ap.add_argument("--expert-cache", type=int, default=0, metavar="SLOTS",
                    help="stream the experts from host memory through a cache of SLOTS experts "
                         "per layer, over a stack of --layers layers (decode batches)")
    ap.add_argument("--layers", type=int, default=16)
    ap.add_argument("--guesses", type=int, default=0,
                    help="experts of the next layer to prefetch, guessed with its router on "
                         "this layer's input (default: top_k)")
    ap.add_argument("--scmoe", action="store_true",
                    help="time the MoE beside sub-block-1's decode attention (shortcut-connected "
                         "MoE): alone, one after the other, and concurrently on two streams")
    ap.add_argument("--context", type=int, default=4096, help="--scmoe: keys per sequence")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), \
        int(os.environ.get("WORLD_SIZE", 1))


def reduce_max(values, device="cpu"):
    """Element-wise maximum of per-rank floats over the process group (each
    rank gets the result); identity without a process group."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world: int, tokens_per_rank: int, max_ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch per step, and the
    job's step lasts as long as the slowest rank's."""
    return world * tokens_per_rank / (max_ms_per_step / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def selected_bytes(fam, counts, fmt: str = "fp8") -> dict:
    """Algorithmic bytes of one step: every active expert's codes and scales
    once, the router, the activations in and out.  fp8: e4m3 codes + one f32
    per 128x128 block; nvfp4: half a byte per weight + one e4m3 per 16
    weights + one f32 per matrix."""
    H, I, E = fam.hidden, fam.inter, fam.n_experts
    n_act = int((np.asarray(counts) > 0).sum())
    if fmt == "nvfp4":
        w13 = 2 * I * H // 2 + 2 * I * H // 16 + 4
        w2 = H * I // 2 + H * I // 16 + 4
    else:
        w13 = 2 * I * H + 4 * (2 * I // 128) * (H // 128)
        w2 = H * I + 4 * (H // 128) * (I // 128)
    return dict(n_active=n_act, w13=n_act * w13, w2=n_act * w2, router=E * H * 4)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"clocks_dev{device}_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.device), "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ oracle timing

def oracle_sample_tokens(fam, T: int) -> int:
    """Tokens of the oracle's bounded sample: the first n tokens of the batch,
    run through the whole layer.  The oracle dequantises every expert the
    sample touches, so the sample is smaller for the large experts."""
    return min(T, 64 if fam.expert_bytes <= (8 << 20) else 8)


_ORACLE_CHILD = r"""
import json, os, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np
import workloads as W
from oracle import threaded
fam, T = W.parse_workload(sys.argv[2])
budget, n, reps_max, warm = float(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5]), int(sys.argv[6])
x = W.make_x(fam, T)[:n]
if sys.argv[7] == "nvfp4":
    from oracle import nvfp4
    w = W.make_weights_fp4(fam)
    run = lambda: nvfp4.moe_forward_nvfp4(x, w.router_w, w.router_bias, w.w13, w.sf13, w.g13,
                                          w.w2, w.sf2, w.g2, fam.top_k)
else:
    w = W.make_weights(fam)
    run = lambda: threaded.moe_forward(x, w.router_w, w.router_bias, w.w13, w.s13, w.w2, w.s2,
                                       fam.top_k)
for _ in range(warm):
    run()
times = []
t0 = time.perf_counter()
while True:
    a = time.perf_counter(); run(); times.append(time.perf_counter() - a)
    if len(times) >= reps_max or (budget > 0 and time.perf_counter() - t0 >= budget):
        break
print(json.dumps({"times": times, "n": n, "T": T,
                  "cores": 1 if sys.argv[7] == "nvfp4" else threaded.default_workers()}))
"""


def _oracle_child(workload: str, budget: float, reps_max: int, warm: int, fmt: str = "fp8") -> dict:
    fam, T = W.parse_workload(workload)
    n = oracle_sample_tokens(fam, T)
    # one expert per thread, each with a single-threaded BLAS
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", _ORACLE_CHILD, ROOT, workload, str(budget), str(n),
                        str(reps_max), str(warm), fmt], capture_output=True, text=True, env=env,
                       timeout=3600)
    if r.returncode != 0:
        raise RuntimeError("oracle run failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def _oracle_sample_text(workload: str, d: dict, fmt: str = "fp8") -> str:
    how = ("FP4 f64 oracle, one thread" if fmt == "nvfp4" else
           f"f64 oracle threaded over tokens (router) and expert segments (FFN) on "
           f"{d['cores']} host threads")
    return (f"whole layer (routing, experts, combine) on the first {d['n']} of the "
            f"{d['T']} tokens of {workload}, {how}; every expert the sample touches is "
            f"dequantised once per pass")


def oracle_rate(workload: str, seconds: float, fmt: str = "fp8") -> dict:
    """Oracle tokens/s on the host cores: passes over the bounded sample for
    about `seconds`, in a fresh process."""
    d = _oracle_child(workload, seconds, 1000, 0, fmt)
    el = sum(d["times"])
    return dict(value=len(d["times"]) * d["n"] / el, unit=UNIT, cores=d["cores"], kind="oracle",
                sample=f"{len(d['times'])} passes, {el:.1f} s: " + _oracle_sample_text(workload, d, fmt),
                seconds=el)


# ------------------------------------------------------------------ native arm

# Source files each dominant kernel is compiled from (its .cu file and the
# headers it includes); a profile's DRAM traffic stays valid while they do not
# change.
KERNEL_SOURCES = {
    "decode_ffn": ("decode_mma.cu", "common.cuh", "kernels.h", "sm100_ptx.cuh"),
    "grouped_gemm": ("prefill_gemm.cu", "common.cuh", "kernels.h", "sm100_ptx.cuh"),
    "gemv": ("gemv.cu", "common.cuh", "kernels.h"),
}


def kernel_source_sha(kernel: str | None = None) -> str:
    """Hash of one kernel's source files (all of csrc/ when kernel is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_routed_expert_gb300", "csrc")
    files = KERNEL_SOURCES[kernel] if kernel else os.listdir(csrc)
    for f in sorted(files):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel's current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(f"{kernel}/{workload}")
    if not e or e.get("source_sha") != kernel_source_sha(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def gemm1_roofline(fam, T: int, sb: dict, launch_s: float, hbm_gbs: float, fp8_tflops: float,
                   peak_src: str) -> dict:
    """Roofline of the gate/up grouped GEMM (one launch, launch_s seconds).

    Algorithmic FLOPs 2 P H 2I; algorithmic bytes = the selected experts' W13
    codes and scales + x (bf16).  Its floor is the larger of bytes / HBM
    bandwidth and FLOPs / FP8 peak; ``bound`` names that side and ``achieved``
    / ``peak`` / ``frac`` are given on it, with the other side beside them
    (``tflops`` / ``fp8_frac`` and ``gbs`` / ``hbm_frac``) and
    ``attainable_frac`` = floor / time."""
    P = T * fam.top_k
    flops = 2.0 * P * fam.hidden * 2 * fam.inter
    nbytes = sb["w13"] + T * fam.hidden * 2
    tflops = flops / launch_s / 1e12
    gbs = nbytes / launch_s / 1e9
    t_hbm, t_tc = nbytes / (hbm_gbs * 1e9), flops / (fp8_tflops * 1e12)
    r = dict(kernel="gate_up_swiglu (grouped GEMM)", algorithmic_flops=flops,
             algorithmic_bytes=nbytes, avg_launch_us=launch_s * 1e6,
             tflops=tflops, fp8_peak_tflops=fp8_tflops, fp8_frac=tflops / fp8_tflops,
             gbs=gbs, hbm_frac=gbs / hbm_gbs, attainable_frac=max(t_hbm, t_tc) / launch_s,
             peak_source=(f"hbm_gbs and bf16_tflops x {FP8_PER_BF16} (nominal fp8/bf16), "
                          f"{peak_src}"))
    if t_hbm >= t_tc:
        r.update(bound="hbm", achieved=gbs, peak=hbm_gbs, unit="GB/s", frac=gbs / hbm_gbs)
    else:
        r.update(bound="tensor", achieved=tflops, peak=fp8_tflops, unit="TFLOP/s",
                 frac=tflops / fp8_tflops)
    return r


def kernel_breakdown(layer, step, flush, dev, n: int):
    """Average CUDA-event time (us) of each kernel step of the layer over n
    extra steps after the timed region (L2 flushed before each).  Events sit
    between the kernels, so the chained launches lose their overlap here; the
    timed region above has no such events.  None if the timing API fails."""
    import torch
    try:
        layer.set_timing("all")
        for _ in range(n):
            flush()
            step()
        torch.cuda.synchronize(dev)
        out = {}
        for name in KERNEL_STEPS:
            ms, c = layer.kernel_time(name)
            if c:
                out[name] = round(ms / c * 1e3, 2)
        layer.set_timing(())
        return out
    except Exception as e:  # the breakdown is auxiliary: never lose the bench line for it
        try:
            layer.set_timing(())
        except Exception:
            pass
        return {"unavailable": str(e)[:200]}


def run_native(args, rank, local_rank, world):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from fp8_routed_expert_gb300 import MoELayer

    fam, T = W.parse_workload(args.workload)
    k = fam.top_k
    fp4 = args.format == "nvfp4"
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.make_weights_fp4(fam) if fp4 else W.make_weights(fam)
    xb = W.make_x(fam, T)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    rw, rb = g(w.router_w), (None if w.router_bias is None else g(w.router_bias))
    if fp4:
        experts = [g(a) for a in (w.w13, w.sf13, w.g13, w.w2, w.sf2, w.g2)]
    else:
        experts = [g(a) for a in (w.w13, w.s13, w.w2, w.s2)]
    x = torch.from_numpy(xb.astype(np.int16)).view(torch.bfloat16).to(dev)
    out = torch.empty_like(x)
    layer = MoELayer(T, fam.hidden, fam.n_experts, fam.inter, k, local_rank)
    layer.set_path(args.path)
    stream = torch.cuda.current_stream(dev)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.max()

    decode = T <= 64
    path = "nvfp4-gemv" if fp4 else layer.resolved_path(T)
    dominant = "gate_up"

    def step():
        if fp4:
            layer.forward_nvfp4(x, rw, rb, *experts, k, out=out, stream=stream)
        else:
            layer.forward(x, rw, rb, *experts, k, out=out, stream=stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    assert layer.status() == 0
    counts = layer.routing(T, k)["counts"].cpu().numpy()

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    layer.set_timing([dominant])
    n0 = layer.launch_count()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        t_wall = time.perf_counter()
        for i in range(K):
            flush()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    launches = layer.launch_count() - n0
    dom_ms, dom_n = layer.kernel_time(dominant)
    layer.set_timing(())
    assert layer.status() == 0
    step_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / K

    kernels_us = kernel_breakdown(layer, step, flush, dev, 20 if decode else 5)

    # end to end with host buffers (pinned): the host-buffer entry point for
    # FP8 experts; for FP4 experts the copies around the device entry point
    xh = torch.from_numpy(xb.astype(np.int16)).view(torch.bfloat16).pin_memory()
    oh = torch.empty_like(xh).pin_memory()

    def e2e_step():
        if fp4:
            x.copy_(xh, non_blocking=True)
            layer.forward_nvfp4(x, rw, rb, *experts, k, out=out, stream=stream)
            oh.copy_(out, non_blocking=True)
        else:
            layer.forward_host(xh, rw, rb, *experts, k, oh, stream=stream)

    for _ in range(3):
        e2e_step()
    K2 = max(1, min(K, 500))
    e2e_ms = []
    for _ in range(K2):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e_step = sum(e2e_ms) / K2

    step_ms, e2e_step = reduce_max([step_ms, e2e_step], device=dev)
    if rank != 0:
        return None

    hbm, bf16, bf16_sus, src = peaks()
    sb = selected_bytes(fam, counts, args.format)
    P = T * k
    dom_s = dom_ms / max(dom_n, 1) / 1e3
    if fp4:
        # gate/up GEMV: selected experts' W13 codes and scales, x (f16) in,
        # h (f32) out
        dom_bytes = sb["w13"] + T * fam.hidden * 2 + P * fam.inter * 4
        achieved = dom_bytes / dom_s / 1e9
        roof = dict(bound="hbm", achieved=achieved, peak=hbm, unit="GB/s", frac=achieved / hbm,
                    traffic=None, kernel="fp4_gate_up (NVFP4 grouped GEMV + SwiGLU)",
                    algorithmic_bytes=dom_bytes, avg_launch_us=dom_s * 1e6,
                    peak_source=f"hbm_gbs, {src}")
    elif decode and path == "tcgemv":
        # one launch streams both projections: selected experts' W13 and W2
        # (codes and scales), the activations in and y out
        dom_bytes = sb["w13"] + sb["w2"] + T * fam.hidden * 2 + P * fam.hidden * 4
        achieved = dom_bytes / dom_s / 1e9
        roof = dict(bound="hbm", achieved=achieved, peak=hbm, unit="GB/s", frac=achieved / hbm,
                    traffic=profiled_traffic("decode_ffn", args.workload),
                    kernel="decode_ffn (tcgen05 gate/up + SwiGLU + down, one launch)",
                    algorithmic_bytes=dom_bytes, avg_launch_us=dom_s * 1e6,
                    peak_source=f"hbm_gbs, {src}")
    elif decode:
        dom_bytes = sb["w13"] + T * fam.hidden * 2 + P * fam.inter * 4
        achieved = dom_bytes / dom_s / 1e9
        roof = dict(bound="hbm", achieved=achieved, peak=hbm, unit="GB/s", frac=achieved / hbm,
                    traffic=profiled_traffic("gemv", args.workload),
                    kernel="gate_up_swiglu (grouped GEMV)", algorithmic_bytes=dom_bytes,
                    avg_launch_us=dom_s * 1e6, peak_source=f"hbm_gbs, {src}")
    else:
        roof = gemm1_roofline(fam, T, sb, dom_s, hbm, bf16 * FP8_PER_BF16, src)
        roof["traffic"] = profiled_traffic("grouped_gemm", args.workload)
    layer_bytes = sb["w13"] + sb["w2"] + sb["router"] + 2 * T * fam.hidden * 2
    layer_gbs = layer_bytes / (step_ms / 1e3) / 1e9
    expert_flops = 6.0 * P * fam.hidden * fam.inter
    fp8_peak = bf16 * FP8_PER_BF16
    layer_floor_s = max(layer_bytes / (hbm * 1e9), expert_flops / (fp8_peak * 1e12))
    value = job_throughput(world, T, step_ms)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("e2m1 (NVFP4) weights x f16 activations, f32 accumulate" if fp4 else
                  "e4m3 weights x f16 activations, f32 accumulate" if path == "gemv" else
                  "e4m3 weights x multi-term e4m3 activations, f32 accumulate"),
        "data": ("synthetic (seeded N(0,1) bf16 activations, N(0,0.02) weights quantised to "
                 + ("NVFP4: e2m1 + e4m3 scale per 16 + f32 per matrix)" if fp4 else
                    "e4m3 per 128x128 block)")),
        "config": {"workload": args.workload, "format": args.format, "tokens": T,
                   "hidden": fam.hidden,
                   "experts": fam.n_experts, "top_k": k, "inter": fam.inter,
                   "active_experts": sb["n_active"],
                   "path": path,
                   "l2": "flushed before every step (256 MiB memset, then a 256 MiB read)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "layer": {"bytes": layer_bytes, "gbs": layer_gbs, "hbm_frac": layer_gbs / hbm,
                  "expert_tflops": expert_flops / (step_ms / 1e3) / 1e12,
                  "expert_fp8_frac": expert_flops / (step_ms / 1e3) / 1e12 / fp8_peak,
                  "attainable_frac": layer_floor_s / (step_ms / 1e3)},
        "gpu_launches": int(launches),
        "kernels_us": kernels_us,
        "e2e": {"value": job_throughput(world, T, e2e_step), "unit": UNIT,
                "h2d_bytes_per_step": T * fam.hidden * 2, "d2h_bytes_per_step": T * fam.hidden * 2,
                "ms_per_step": e2e_step},
        "wall_s_timed_region": t_wall,
        "clocks": clk.summary(),
    }
    return res


def run_stream(args) -> dict:
    """Decode through a stack of layers whose experts live in host memory.

    Layer l has its own seeded weights (seed * 100 + l); x_{l+1} = x_l +
    MoE_l(x_l).  Three ways are timed over the same token batches: every
    expert resident in device memory; the expert cache (SLOTS per layer,
    copies over NVLink-C2C when an expert is missing); the cache with the
    next layer's experts guessed from its router on this layer's input and
    prefetched while this layer computes."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from fp8_routed_expert_gb300 import ExpertCache, MoELayer

    fam, T = W.parse_workload(args.workload)
    k, L, slots = fam.top_k, args.layers, args.expert_cache
    n_guess = args.guesses or k
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    layers = []
    for l in range(L):
        f = W.Family(fam.name, fam.hidden, fam.n_experts, fam.top_k, fam.inter, fam.seed * 100 + l,
                     fam.tokens, fam.bias_std)
        w = W.make_weights(f)
        layers.append(dict(
            rw=g(w.router_w), rb=None if w.router_bias is None else g(w.router_bias),
            s13=g(w.s13), s2=g(w.s2),
            # page-locked buffers allocated by the CUDA driver (placed for the
            # GPU's host link), as an engine loading the experts would use
            w13_host=torch.from_numpy(w.w13).pin_memory(), w2_host=torch.from_numpy(w.w2).pin_memory(),
            w13=g(w.w13), w2=g(w.w2),
            ctx=MoELayer(T, fam.hidden, fam.n_experts, fam.inter, k, 0)))
    for ly in layers:
        ly["cache"] = ExpertCache(ly["ctx"], ly["w13_host"], ly["w2_host"], slots)
    xs = [torch.from_numpy(W.normal_bf16(9000 + i, W.configs.TID_X, (T, fam.hidden)).astype(np.int16))
          .view(torch.bfloat16).to(dev) for i in range(args.steps + args.warmup)]

    def token_step(x, mode):
        for l, ly in enumerate(layers):
            if mode == "resident":
                out = ly["ctx"].forward(x, ly["rw"], ly["rb"], ly["w13"], ly["s13"], ly["w2"],
                                        ly["s2"], k, stream=stream)
            else:
                out = ly["cache"].forward(x, ly["rw"], ly["rb"], ly["s13"], ly["s2"], k, stream=stream)
                if mode == "prefetch" and l + 1 < L:
                    nxt = layers[l + 1]
                    nxt["cache"].prefetch(nxt["cache"].guess(x, nxt["rw"], nxt["rb"], k, n_guess))
            x = x + out
        return x

    res = {}
    for mode in ("resident", "cache", "prefetch"):
        before = [ly["cache"].stats() for ly in layers]
        for i in range(args.warmup):
            token_step(xs[i], mode)
        torch.cuda.synchronize(dev)
        mid = [ly["cache"].stats() for ly in layers]
        t0 = time.perf_counter()
        for i in range(args.steps):
            token_step(xs[args.warmup + i], mode)
        torch.cuda.synchronize(dev)
        el = time.perf_counter() - t0
        after = [ly["cache"].stats() for ly in layers]
        d = {key: sum(a[key] - m[key] for a, m in zip(after, mid)) for key in after[0]}
        res[mode] = dict(tokens_s=T * args.steps / el, ms_per_token_step=el / args.steps * 1e3,
                         **{f"{kk}": v for kk, v in d.items()})
        del before
    hbm, _, _, src = peaks()
    pf, ca = res["prefetch"], res["cache"]
    lookups = lambda r: r["hits"] + r["misses"]
    return {
        "metric": METRIC, "value": pf["tokens_s"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": pf["ms_per_token_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 weights x multi-term e4m3 activations, f32 accumulate",
        "data": "synthetic (seeded per layer; a new token batch every step)",
        "config": {"workload": f"{args.workload} through {L} layers, experts in host memory",
                   "layers": L, "slots_per_layer": slots, "experts_per_layer": fam.n_experts,
                   "guesses": n_guess, "expert_bytes": 3 * fam.hidden * fam.inter,
                   "host_expert_bytes": L * fam.n_experts * 3 * fam.hidden * fam.inter},
        "stream": {
            "resident_tokens_s": res["resident"]["tokens_s"],
            "cache_tokens_s": ca["tokens_s"], "cache_prefetch_tokens_s": pf["tokens_s"],
            "cache_hit_rate": ca["hits"] / max(lookups(ca), 1),
            "prefetch_hit_rate": pf["hits"] / max(lookups(pf), 1),
            "prefetched_used_frac": pf["prefetch_used"] / max(pf["prefetched"], 1),
            "c2c_gbs_cache": ca["bytes_copied"] / (ca["ms_per_token_step"] * args.steps / 1e3) / 1e9,
            "c2c_gbs_prefetch": pf["bytes_copied"] / (pf["ms_per_token_step"] * args.steps / 1e3) / 1e9,
            "per_mode": res},
    }


def run_scmoe(args) -> dict:
    """Shortcut-connected MoE overlap.  The MoE runs on sub-block-0's output
    while sub-block-1's attention (one new token per sequence over a cache of
    --context keys, heads = H / 128) runs on another stream; the MoE's
    persistent kernels get an SM budget so that the attention finds free SMs.
    Reported: each alone, one after the other, and overlapped (best budget)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from fp8_routed_expert_gb300 import MoELayer, lib

    fam, T = W.parse_workload(args.workload)
    k, S = fam.top_k, args.context
    nh = fam.hidden // 128
    dev = torch.device("cuda", 0)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda bits: torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(dev)
    w = W.make_weights(fam)
    rw, rb = g(w.router_w), (None if w.router_bias is None else g(w.router_bias))
    w13, s13, w2, s2 = g(w.w13), g(w.s13), g(w.w2), g(w.s2)
    x = bf(W.make_x(fam, T))
    q = bf(W.normal_bf16(77, 11, (T, nh, 128)))
    kc = bf(W.normal_bf16(77, 12, (T, S, nh, 128)))
    vc = bf(W.normal_bf16(77, 13, (T, S, nh, 128)))
    att = torch.empty_like(q)
    ws = torch.empty(lib().moe_attention_workspace_bytes(T, S, nh, 128), dtype=torch.uint8, device=dev)
    moe_out = torch.empty_like(x)
    layer = MoELayer(T, fam.hidden, fam.n_experts, fam.inter, k, 0)
    # the MoE's stream has the higher priority: its short routing kernels and
    # its expert kernels are scheduled ahead of waiting attention CTAs
    lo, hi = torch.cuda.Stream.priority_range() if hasattr(torch.cuda.Stream, "priority_range") \
        else (0, -1)
    sa, sb = torch.cuda.Stream(dev, priority=hi), torch.cuda.Stream(dev, priority=lo)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def moe(st):
        layer.forward(x, rw, rb, w13, s13, w2, s2, k, out=moe_out, stream=st)

    def attn(st):
        rc = lib().moe_decode_attention(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), T, S, nh, nh, 128,
                                        att.data_ptr(), ws.data_ptr(), ws.numel(), st.cuda_stream)
        assert rc == 0

    def timed(fn, reps):
        ms = []
        for _ in range(reps):
            flush_w.zero_()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(sa)
            fn()
            ev = torch.cuda.Event()
            ev.record(sb)
            sa.wait_event(ev)
            b.record(sa)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.median(ms) * 1e3

    def serial():
        moe(sa)
        attn(sa)

    def overlapped():
        ev = torch.cuda.Event()
        ev.record(sa)
        sb.wait_event(ev)
        moe(sa)
        attn(sb)

    reps = max(args.steps, 20)
    for fn in (lambda: moe(sa), lambda: attn(sa), serial, overlapped):
        timed(fn, 3)
    # the same with the experts streamed from host memory through an expert
    # cache: the copies of missing experts (copy engine, no SMs) can run
    # under the attention -- the pages' point of the overlap window
    from fp8_routed_expert_gb300 import ExpertCache
    slots = args.expert_cache or min(fam.n_experts, 48)
    cache = ExpertCache(layer, torch.from_numpy(w.w13).pin_memory(), torch.from_numpy(w.w2).pin_memory(),
                        slots)
    xs = [bf(W.normal_bf16(9500 + i, W.configs.TID_X, (T, fam.hidden))) for i in range(4 * reps + 40)]
    it = iter(xs)

    def moe_cached(st):
        cache.forward(next(it), rw, rb, s13, s2, k, out=moe_out, stream=st)

    def serial_cached():
        attn(sa)
        moe_cached(sa)

    def overlapped_cached():
        ev = torch.cuda.Event()
        ev.record(sa)
        sb.wait_event(ev)
        attn(sb)          # enqueued first: runs while the MoE routes and copies
        moe_cached(sa)

    for fn in (lambda: moe_cached(sa), serial_cached, overlapped_cached):
        timed(fn, 3)
    cached = {"slots": slots, "moe_us": timed(lambda: moe_cached(sa), reps),
              "serial_us": timed(serial_cached, reps), "overlapped_us": timed(overlapped_cached, reps)}
    cached["saved_frac"] = 1 - cached["overlapped_us"] / cached["serial_us"]
    cache.close()
    res = {"moe_us": timed(lambda: moe(sa), reps), "attention_us": timed(lambda: attn(sa), reps),
           "serial_us": timed(serial, reps)}
    budgets = {}
    for budget in (0, 136, 120, 104, 88):
        lib().moe_set_sm_budget(layer.handle, budget)
        timed(overlapped, 3)
        budgets[str(budget or "all")] = timed(overlapped, reps)
    lib().moe_set_sm_budget(layer.handle, 0)
    best = min(budgets, key=budgets.get)
    res.update(overlapped_us_by_moe_sm_budget=budgets, best_budget=best,
               overlapped_us=budgets[best], saved_frac=1 - budgets[best] / res["serial_us"],
               streamed_experts=cached)
    kv_bytes = 2 * T * S * nh * 128 * 2
    return {"metric": METRIC, "value": T / (budgets[best] / 1e6), "unit": UNIT, "n_gpus": 1,
            "steps": reps, "warmup": 3, "ms_per_step": budgets[best] / 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 weights x multi-term e4m3 activations, f32 accumulate; bf16 attention",
            "data": "synthetic", "config": {"workload": f"{args.workload} beside decode attention",
                                             "context": S, "heads": nh, "kv_bytes": kv_bytes,
                                             "l2": "flushed before every rep"},
            "scmoe": res}


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    fam, T = W.parse_workload(args.workload)
    if args.impl == "reference":
        if rank != 0:
            return 0
        steps = args.steps if args.steps is not None else 3
        warm = args.warmup if args.warmup is not None else 1
        r = oracle_reference_arm(args.workload, steps, warm)
        r.update(n_gpus=args.gpus, steps=steps, warmup=warm)
        print(json.dumps(r))
        return 0

    if args.scmoe:
        args.steps = args.steps or 50
        print(json.dumps(run_scmoe(args)))
        return 0
    if args.expert_cache:
        args.steps = args.steps or 50
        args.warmup = max(args.warmup or 5, 3)
        print(json.dumps(run_stream(args)))
        return 0
    if args.steps is None:
        args.steps = 3000 if T <= 64 else 200
    if args.warmup is None:
        args.warmup = 20
    args.warmup = max(args.warmup, 3)
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = run_native(args, rank, local_rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = oracle_rate(args.workload, args.cpu_seconds, args.format)
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


def oracle_reference_arm(workload: str, steps: int, warmup: int) -> dict:
    """The reference arm: the CPU oracle timed on the host cores, one bounded
    sample of the workload per step (the whole layer on the batch's first
    tokens, threaded over tokens and expert segments)."""
    try:
        d = _oracle_child(workload, 0.0, steps, warmup)
    except Exception as e:  # noqa: BLE001
        return {"impl": "reference", "unavailable": str(e)[-300:]}
    times = d["times"][:steps]
    sec = sum(times) / len(times)
    value = d["n"] / sec
    fam, T = W.parse_workload(workload)
    sample = "per step: " + _oracle_sample_text(workload, d)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload, "tokens": T, "hidden": fam.hidden,
                       "experts": fam.n_experts, "top_k": fam.top_k, "inter": fam.inter},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": d["cores"], "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


if __name__ == "__main__":
    sys.exit(main())
