#!/usr/bin/env python
"""Benchmark of the block-scaled FP4 hot path on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one pass of the whole hot path over one batch of synthetic input.
For the default workload, the LLM MLP up-projection (BF16 activations
16384x8192 ~N(0,1) and weights 28672x8192 ~N(0,0.015), quantized to MXFP4 and
multiplied, BF16 out), a step is: one grouped quantize of A and W (scales
written straight into the tcgen05 tile order), then the GEMM.  `value` is
2*M*N*K per step over the device time of the step, in TFLOP/s; the GEMM
kernel alone and the quantizer's GB/s are reported beside it with their
roofline fractions: against the measured burst bf16 rate times the nominal
FP4:BF16 ratio, and, per clock, against the FP4 MMA rate this GPU is
calibrated at in the same run (mx_calibrate_mma) at the SM clock sampled
while the kernel ran.  The quantize-only workloads (quant2d_*: a
bidimensional MXFP4 quantize; nvfp4_sr_*: an NVFP4 quantize with stochastic
rounding; nvfp4_quant2d_sr_*: both; nvfp4_quant2d_*: bidimensional NVFP4 with
rounding to nearest) have no GEMM and report GB/s of algorithmic bytes instead.

Timing: inputs are resident in HBM; the K steps are replayed from CUDA graphs
(each holding one step per rotating input set) between two CUDA events on the
launching stream,
with enough rotating sets that the working set exceeds 3x the L2 (129 MB),
so every step reads cold operands.  Per-kernel durations come from CUDA
events around graphs of back-to-back launches of each call over the same
rotating sets.  SM clocks and throttle reasons are sampled with nvidia-smi
during the timed region.

`e2e` is the same metric through the public C ABI with the inputs in pinned
host memory: every step copies A and W host->device, quantizes, multiplies
and copies D back, with the steps pipelined over three streams (copy in,
compute, copy out) so that one step's copies overlap its neighbours' compute.  `cpu_baseline` is the CPU oracle (tests' reference
implementation, untuned) on a bounded sample of the same step.

--impl reference times that oracle instead (rank 0 only), each step a
bounded sample sized so the whole run takes a few minutes.

Multi-GPU: the workload has no exchange step, so N GPUs run N independent
replicas (weak scaling); the step time is the max over ranks and `value`
sums the work of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from block_scaled_fp4_bf16_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "mlp_up_16384x28672x8192"
METRIC = "MXFP4 GEMM TFLOPS and % of GB300 dense FP4 peak; quantize GB/s vs HBM"

# Steps with no GEMM (a quantize alone, or the FP4 code transpose): their
# metric is algorithmic GB/s.
QUANT_KINDS = ("quant2d", "quant_sr", "transpose")
# Philox seed of the stochastic-rounding quantize step
SR_SEED = 0x5EED5EED


def quant_step_bytes(w, m, k):
    """Algorithmic bytes of a step without a GEMM (workload w) over an [m, k]
    tensor: a quantize of BF16, or the transpose of FP4 codes."""
    if w["kind"] == "transpose":            # codes read once, written once
        return m * k * (0.5 + 0.5)
    nv = w["fmt"] == "nvfp4"
    amax = 2 if nv else 0                   # NVFP4: the amax pass reads x once more
    blk = 16 if nv else 32
    if w["kind"] == "quant2d":              # x read once; codes + scales of x and of x^T
        return m * k * (amax + 2 + 2 * (0.5 + 1.0 / blk))
    return m * k * (amax + 2 + 0.5 + 1.0 / blk)
L2_BYTES = 129 * 1024 * 1024
FP4_OVER_BF16 = 13.5 / 2.25   # nominal dense FP4 : BF16 tensor ratio on GB300
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------- setup

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=synth.WORKLOAD_ORDER)
    p.add_argument("--e2e-steps", type=int, default=None)
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--min-call-seconds", type=float, default=1.5,
                   help="least time each call's own timing loop runs (0 for runs under ncu)")
    p.add_argument("--calibrate", action="store_true",
                   help="print the FP4 MMA rate of every form and shape (mx_calibrate_mma), "
                        "one JSON line each, and exit")
    a = p.parse_args(argv)
    a.warmup = max(a.warmup, 3)
    a.steps = max(a.steps, 1)
    return a


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x, world, device):
    """The maximum of a per-rank float over all ranks of the default process
    group (x itself on one rank); device: where the collective's tensor lives
    ("cuda" under NCCL, "cpu" under gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(work_per_step, ms_per_step_max, world):
    """Whole-job throughput of N replicas: every rank does work_per_step per
    step, and the job's step takes the slowest rank's time."""
    return world * work_per_step / (ms_per_step_max * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def workload_shape(name):
    w = synth.WORKLOADS[name]
    return w, w["m"], w["n"], w["k"]


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons (background)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str, interval_ms: int = 100):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(interval_ms), "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append((time.time(), float(parts[1]), float(parts[2]),
                                     parts[5:9]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside:   # timed region shorter than the sampling period
            inside = [s for s in self.samples if t0 - 1.0 <= s[0] <= t1 + 0.2]
            window = "timed region +- sampling period (region shorter than one sample)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no samples"}
        reasons = sorted({self.NAMES[i] for s in inside for i, v in enumerate(s[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# --------------------------------------------------------------------- device workload

class DeviceWorkload:
    """Device buffers of one workload (several rotating input sets) and its step."""

    def __init__(self, name: str, host_inputs: dict, nsets: int):
        import torch
        import block_scaled_fp4_bf16_gb300 as mx
        self.mx = mx
        self.torch = torch
        self.name = name
        self.w, self.m, self.n, self.k = workload_shape(name)
        w, m, n, k = self.w, self.m, self.n, self.k
        self.fmt = mx.MX_FMT_MXFP4 if w["fmt"] == "mxfp4" else mx.MX_FMT_NVFP4
        self.out = mx.MX_OUT_BF16 if w["out"] == "bf16" else mx.MX_OUT_FP32
        self.kind = w["kind"]
        self.split_k = w["split_k"]
        self.sets = []
        dev = "cuda"
        u8 = torch.uint8
        sa_bytes = mx.mx_scale_bytes(m, k, self.fmt, mx.MX_SCALE_TCGEN05)
        sb_bytes = mx.mx_scale_bytes(n, k, self.fmt, mx.MX_SCALE_TCGEN05) if n else 0
        wsb = mx.mx_gemm_workspace_bytes(m, n, k, self.split_k) if n else 0
        out_dt = torch.bfloat16 if self.out == mx.MX_OUT_BF16 else torch.float32
        if self.kind == "bf16":
            ha = torch.from_numpy(host_inputs["a"].view(np.int16)).view(torch.bfloat16)
            hb = torch.from_numpy(host_inputs["b"].view(np.int16)).view(torch.bfloat16)
        elif self.kind == "transpose":
            hc = torch.from_numpy(host_inputs["a_codes"])
        elif self.kind in QUANT_KINDS:
            ha = torch.from_numpy(host_inputs["a"].view(np.int16)).view(torch.bfloat16)
        else:
            tiled = {}
            for key, rows in (("a", m), ("b", n)):
                plain = torch.from_numpy(host_inputs[f"{key}_scales"]).to(dev)
                t = torch.empty(mx.mx_scale_bytes(rows, k, self.fmt, mx.MX_SCALE_TCGEN05),
                                dtype=u8, device=dev)
                mx.mx_scale_relayout(plain, rows, k, self.fmt, t)
                tiled[key] = t
        for _ in range(nsets):
            s = {}
            if self.kind == "transpose":
                s["codes_in"] = hc.to(dev)
                s["codes_t"] = torch.empty(m * k // 2, dtype=u8, device=dev)
                self.sets.append(s)
                continue
            if self.kind == "quant2d":
                s["x_a"] = ha.to(dev)
                s["codes_a"] = torch.empty(m * k // 2, dtype=u8, device=dev)
                s["sf_a"] = torch.empty(sa_bytes, dtype=u8, device=dev)
                s["codes_t"] = torch.empty(m * k // 2, dtype=u8, device=dev)
                s["sf_t"] = torch.empty(mx.mx_scale_bytes(k, m, self.fmt, mx.MX_SCALE_TCGEN05),
                                        dtype=u8, device=dev)
                if self.fmt == mx.MX_FMT_NVFP4:
                    s["ts_a"] = torch.zeros(1, dtype=torch.float32, device=dev)
                    s["qws"] = torch.empty(mx.mx_quantize_workspace_bytes(m, k, self.fmt),
                                           dtype=u8, device=dev)
                self.sets.append(s)
                continue
            if self.kind == "quant_sr":
                s["x_a"] = ha.to(dev)
                s["codes_a"] = torch.empty(m * k // 2, dtype=u8, device=dev)
                s["sf_a"] = torch.empty(sa_bytes, dtype=u8, device=dev)
                s["ts_a"] = torch.zeros(1, dtype=torch.float32, device=dev)
                s["qws"] = torch.empty(mx.mx_quantize_workspace_bytes(m, k, self.fmt), dtype=u8,
                                       device=dev)
                self.sets.append(s)
                continue
            if self.kind == "bf16":
                s["x_a"] = ha.to(dev)
                s["x_b"] = hb.to(dev)
                s["codes_a"] = torch.empty(m * k // 2, dtype=u8, device=dev)
                s["codes_b"] = torch.empty(n * k // 2, dtype=u8, device=dev)
                s["sf_a"] = torch.empty(sa_bytes, dtype=u8, device=dev)
                s["sf_b"] = torch.empty(sb_bytes, dtype=u8, device=dev)
                if self.fmt == mx.MX_FMT_NVFP4:
                    s["ts_a"] = torch.zeros(1, dtype=torch.float32, device=dev)
                    s["ts_b"] = torch.zeros(1, dtype=torch.float32, device=dev)
                    qws = mx.mx_quantize_group_workspace_bytes(2, self.fmt)
                    s["qws"] = torch.empty(qws, dtype=u8, device=dev)
                if "bias" in host_inputs:
                    s["bias"] = torch.from_numpy(host_inputs["bias"]).to(dev)
            else:
                s["codes_a"] = torch.from_numpy(host_inputs["a_codes"]).to(dev)
                s["codes_b"] = torch.from_numpy(host_inputs["b_codes"]).to(dev)
                s["sf_a"] = tiled["a"].clone()
                s["sf_b"] = tiled["b"].clone()
            s["d"] = torch.empty((m, n), dtype=out_dt, device=dev)
            s["ws"] = torch.empty(wsb, dtype=u8, device=dev) if wsb else None
            self.sets.append(s)
        self.set_bytes = sum(t.numel() * t.element_size() for t in self.sets[0].values()
                             if t is not None)
        torch.cuda.synchronize()

    # The C-ABI calls of one step, in order: (label, callable(set, stream)).
    def calls(self):
        mx = self.mx
        m, n, k, fmt = self.m, self.n, self.k, self.fmt
        out = []
        if self.kind == "transpose":
            def tr(s, st):
                mx.mx_fp4_transpose(s["codes_in"], m, k, s["codes_t"], stream=st)
            return [("transpose", tr)]
        if self.kind == "quant2d" and fmt == mx.MX_FMT_NVFP4:
            sr = 1 if self.w.get("sr") else 0

            def qnv2d(s, st):
                mx.nvfp4_quantize_bf16_2d(s["x_a"], m, k, k, mx.MX_SCALE_TCGEN05, s["codes_a"],
                                          s["sf_a"], s["codes_t"], s["sf_t"], s["ts_a"], sr,
                                          SR_SEED, 10, s["qws"], stream=st)
            return [("quantize_2d", qnv2d)]
        if self.kind == "quant2d":
            def q2d(s, st):
                mx.mx_quantize_bf16_2d(s["x_a"], m, k, k, fmt, mx.MX_SCALE_TCGEN05, s["codes_a"],
                                       s["sf_a"], s["codes_t"], s["sf_t"], stream=st)
            return [("quantize_2d", q2d)]
        if self.kind == "quant_sr":
            def qsr(s, st):
                mx.nvfp4_quantize_bf16_sr(s["x_a"], m, k, k, mx.MX_SCALE_TCGEN05, s["codes_a"],
                                          s["sf_a"], s["ts_a"], SR_SEED, 10, s["qws"], stream=st)
            return [("quantize_sr", qsr)]
        if self.kind == "bf16":
            # the activation and the weight in one grouped quantize call
            def q(s, st):
                mx.mx_quantize_bf16_group(
                    [(s["x_a"], m, k, k, s["codes_a"], s["sf_a"], s.get("ts_a")),
                     (s["x_b"], n, k, k, s["codes_b"], s["sf_b"], s.get("ts_b"))],
                    fmt, mx.MX_SCALE_TCGEN05, s.get("qws"), stream=st)
            out.append(("quantize", q))

        gelu = bool(self.w.get("gelu"))

        def gemm(s, st):
            if fmt == mx.MX_FMT_MXFP4 and (gelu or "bias" in s):
                mx.mxfp4_gemm_ex(s["codes_a"], s["sf_a"], s["codes_b"], s["sf_b"], s["d"], m, n, k,
                                 mx.MX_LAYOUT_TN, self.out, self.split_k, s.get("bias"), 0.0, gelu,
                                 s["ws"], stream=st)
            elif fmt == mx.MX_FMT_MXFP4:
                mx.mxfp4_gemm(s["codes_a"], s["sf_a"], s["codes_b"], s["sf_b"], s["d"], m, n, k,
                              mx.MX_LAYOUT_TN, self.out, self.split_k, s["ws"], stream=st)
            else:
                mx.nvfp4_gemm(s["codes_a"], s["sf_a"], s["codes_b"], s["sf_b"], s["ts_a"],
                              s["ts_b"], s["d"], m, n, k, mx.MX_LAYOUT_TN, self.out,
                              self.split_k, s["ws"], stream=st)
        out.append(("gemm", gemm))
        return out

    def kernels_per_call(self):
        """Kernel launches of each call of the step (matches the library's launches)."""
        mx = self.mx
        if self.kind == "transpose":
            return {"transpose": 1}
        if self.kind == "quant2d":
            return {"quantize_2d": 1 if self.fmt == mx.MX_FMT_MXFP4 else 2}
        if self.kind == "quant_sr":
            return {"quantize_sr": 2}
        q = 1 if self.fmt == mx.MX_FMT_MXFP4 else 2
        g = 1 + (1 if mx.mx_gemm_workspace_bytes(self.m, self.n, self.k, self.split_k) else 0)
        res = {"gemm": g}
        if self.kind == "bf16":
            res["quantize"] = q
        return res

    def algorithmic(self):
        """Algorithmic work of each call: (bytes, flops)."""
        m, n, k = self.m, self.n, self.k
        blk = 32 if self.fmt == self.mx.MX_FMT_MXFP4 else 16
        if self.kind == "transpose":
            return {"transpose": (quant_step_bytes(self.w, m, k), 0.0)}
        if self.kind == "quant2d":
            # BF16 read once, codes and scales written for x and for x^T
            return {"quantize_2d": (quant_step_bytes(self.w, m, k), 0.0)}
        if self.kind == "quant_sr":
            return {"quantize_sr": (quant_step_bytes(self.w, m, k), 0.0)}
        amax_pass = 0 if self.fmt == self.mx.MX_FMT_MXFP4 else 2
        qbytes = lambda r: r * k * (2 + amax_pass + 0.5 + 1.0 / blk)
        out_b = 2 if self.out == self.mx.MX_OUT_BF16 else 4
        gemm_bytes = (m + n) * k * (0.5 + 1.0 / blk) + m * n * out_b
        if self.w.get("bias"):
            gemm_bytes += n * 4
        res = {"gemm": (gemm_bytes, 2.0 * m * n * k)}
        if self.kind == "bf16":
            res["quantize"] = (qbytes(m) + qbytes(n), 0.0)
        return res

    def step(self, i, stream):
        s = self.sets[i % len(self.sets)]
        for _, fn in self.calls():
            fn(s, stream)


# --------------------------------------------------------------------- timing (ours)

def capture_steps(wl, stream, first, count):
    """One CUDA graph of `count` consecutive steps over the rotating sets."""
    torch = wl.torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(first, first + count):
            wl.step(i, h)
    return g


def time_graphs(wl, steps, warmup):
    """Headline set-up: the K steps are issued as replays of a graph holding one
    pass over all rotating sets (plus one graph for the K mod sets remainder),
    so kernels of consecutive steps overlap through programmatic dependent
    launch as they would in a production loop."""
    torch = wl.torch
    stream = torch.cuda.Stream()
    nsets = len(wl.sets)
    for i in range(nsets):
        wl.step(i, torch.cuda.current_stream().cuda_stream)   # eager warm-up of every set
    torch.cuda.synchronize()
    full = capture_steps(wl, stream, 0, nsets)
    rem = steps % nsets
    part = capture_steps(wl, stream, 0, rem) if rem else None
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-warmup // nsets))):
            full.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    return (full, part), stream, start, end


def run_graph_region(wl, graphs, stream, start, end, steps, barrier):
    """Exactly `steps` steps between two events on the launching stream."""
    torch = wl.torch
    full, part = graphs
    nsets = len(wl.sets)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps // nsets):
            full.replay()
        if part is not None:
            part.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    return start.elapsed_time(end), t0, t1


def time_calls(wl, steps, per_graph=40, windows=None, min_seconds=1.5):
    """Per-call device durations: for each C-ABI call of the step, a CUDA graph of
    `per_graph` back-to-back calls over the rotating sets, replayed between two
    events on the launching stream (no host gaps); returns ms per call.
    windows (dict, optional) receives each call's (t0, t1) host-time window, for
    the clock samples taken while it ran; each call is then replayed for at
    least min_seconds, so that the window holds a dozen or more samples and the
    clock has settled under the power limit."""
    torch = wl.torch
    stream = torch.cuda.Stream()
    out = {}
    for label, fn in wl.calls():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            h = torch.cuda.current_stream().cuda_stream
            for i in range(per_graph):
                fn(wl.sets[i % len(wl.sets)], h)
        reps = max(2, steps // per_graph)
        with torch.cuda.stream(stream):
            w0 = torch.cuda.Event(enable_timing=True)
            w1 = torch.cuda.Event(enable_timing=True)
            w0.record(stream)
            g.replay()
            g.replay()
            w1.record(stream)
        torch.cuda.synchronize()
        if windows is not None:
            per_replay = max(w0.elapsed_time(w1) * 1e-3 / 2, 1e-6)
            reps = max(reps, int(math.ceil(min_seconds / per_replay)))
        t0 = time.time()
        with torch.cuda.stream(stream):
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for _ in range(reps):
                g.replay()
            end.record(stream)
        torch.cuda.synchronize()
        if windows is not None:
            windows[label] = (t0, time.time())
        out[label] = start.elapsed_time(end) / (reps * per_graph)
        del g
    return out


def time_e2e(wl, host_inputs, steps):
    """Same metric through the C ABI from pinned host buffers: every step copies
    its inputs host -> device, runs the step's calls and copies its result back
    to the host.  The steps are pipelined over three streams (copy in, compute,
    copy out), as a serving loop would run them: step i's inputs are copied
    while step i-1 computes and step i-2's result is read back.  A rotating set's
    device buffers are refilled only after the step that last used them has been
    read back, and each set has its own pinned result buffers."""
    torch = wl.torch
    pinned = {}
    if wl.kind == "transpose":
        pinned["codes_in"] = torch.from_numpy(host_inputs["a_codes"]).pin_memory()
    elif wl.kind in ("bf16",) + QUANT_KINDS:
        pinned["x_a"] = torch.from_numpy(host_inputs["a"].view(np.int16)).view(
            torch.bfloat16).pin_memory()
    if wl.kind == "bf16":
        pinned["x_b"] = torch.from_numpy(host_inputs["b"].view(np.int16)).view(
            torch.bfloat16).pin_memory()
        if "bias" in host_inputs:
            pinned["bias"] = torch.from_numpy(host_inputs["bias"]).pin_memory()
    elif wl.kind == "codes":
        pinned["codes_a"] = torch.from_numpy(host_inputs["a_codes"]).pin_memory()
        pinned["codes_b"] = torch.from_numpy(host_inputs["b_codes"]).pin_memory()
    # the step's result read back: D, or the code outputs of a quantize step
    result_keys = {"quant2d": ["codes_a", "codes_t"], "quant_sr": ["codes_a"],
                   "transpose": ["codes_t"]}.get(wl.kind, ["d"])
    nset = len(wl.sets)
    results = [{key: torch.empty(st[key].shape, dtype=st[key].dtype).pin_memory()
                for key in result_keys} for st in wl.sets]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in results[0].values())
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_out = {}

    def one(i):
        k = i % nset
        st = wl.sets[k]
        if i - nset in ev_out:
            s_in.wait_event(ev_out.pop(i - nset))  # set k's last step has been read back
        with torch.cuda.stream(s_in):
            for key, t in pinned.items():
                st[key].view(-1).copy_(t.view(-1), non_blocking=True)
        ev_in = torch.cuda.Event()
        ev_in.record(s_in)
        s_cmp.wait_event(ev_in)
        for _, fn in wl.calls():
            fn(st, s_cmp.cuda_stream)
        ev_cmp = torch.cuda.Event()
        ev_cmp.record(s_cmp)
        s_out.wait_event(ev_cmp)
        with torch.cuda.stream(s_out):
            for key, t in results[k].items():
                t.copy_(st[key], non_blocking=True)
        ev_out[i] = torch.cuda.Event()
        ev_out[i].record(s_out)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    ev_out.clear()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        one(i)
    end.record(s_out)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, h2d, d2h


# --------------------------------------------------------------------- CPU oracle

def oracle_step_sample(name, host, frac, prepared):
    """Run the CPU oracle on the fraction `frac` of one step; returns (seconds,
    the fraction actually run).  Quantize-only steps take the first rows of
    the tensor.  GEMM steps take a sqrt(frac) M x sqrt(frac) N block of D
    (every output of it over the whole K) and quantize the matching share
    (frac) of the rows of A and of B, so that each part of the step is cut
    by the same factor."""
    import oracle
    w, m, n, k = workload_shape(name)
    mr = max(1, int(round(m * frac)))
    nr = max(1, int(round(n * frac)))
    g = math.sqrt(frac)
    dm = max(1, min(m, int(round(m * g))))     # output rows of the block
    dn = max(1, min(n, int(round(n * g))))     # output columns of the block
    t0 = time.perf_counter()
    if w["kind"] == "quant2d":
        mr = max(32, mr // 32 * 32)
        if w["fmt"] == "nvfp4":
            oracle.nvfp4_quantize_2d(host["a"][:mr], seed=SR_SEED if w.get("sr") else None)
        else:
            oracle.mx_quantize_2d(host["a"][:mr])
        return time.perf_counter() - t0, mr / m
    if w["kind"] == "quant_sr":
        oracle.nvfp4_quantize_sr(host["a"][:mr], SR_SEED, 10)
        return time.perf_counter() - t0, mr / m
    if w["kind"] == "transpose":
        mr = max(32, mr // 32 * 32)
        oracle.fp4_transpose(host["a_codes"][:mr], mr, k)
        return time.perf_counter() - t0, mr / m
    rows, cols = np.arange(dm), np.arange(dn)
    if w["kind"] == "bf16":
        if w["fmt"] == "mxfp4":
            oracle.mx_quantize(host["a"][:mr])
            oracle.mx_quantize(host["b"][:nr])
            qa, sa, qb, sb = prepared
            d = oracle.mx_gemm(qa, sa, qb, sb, m, n, k, rows=rows, cols=cols)[0]
            if w.get("bias") or w.get("gelu"):
                bias = host.get("bias")
                oracle.gemm_epilogue(d, bias=None if bias is None else bias[:dn],
                                     gelu_on=bool(w.get("gelu")))
        else:
            oracle.nvfp4_quantize(host["a"][:mr])
            oracle.nvfp4_quantize(host["b"][:nr])
            qa, sa, ta, qb, sb, tb = prepared
            oracle.nvfp4_gemm(qa, sa, qb, sb, m, n, k, ta, tb, rows=rows, cols=cols)
    else:
        oracle.mx_gemm(host["a_codes"], host["a_scales"], host["b_codes"], host["b_scales"],
                       m, n, k, rows=rows, cols=cols)
    return time.perf_counter() - t0, dm * dn / (m * n)


def oracle_prepare(name, host):
    import oracle
    w = synth.WORKLOADS[name]
    if w["kind"] not in ("bf16",):
        return None
    if w["fmt"] == "mxfp4":
        qa, sa = oracle.mx_quantize(host["a"])
        qb, sb = oracle.mx_quantize(host["b"])
        return qa, sa, qb, sb
    qa, sa, ta = oracle.nvfp4_quantize(host["a"])
    qb, sb, tb = oracle.nvfp4_quantize(host["b"])
    return qa, sa, ta, qb, sb, tb


def oracle_threads():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else (os.cpu_count() or 1)


def cpu_baseline(name, host, target_s):
    """Bounded sample of the step on the CPU oracle, scaled to the metric."""
    _, m, n, k = workload_shape(name)
    prepared = oracle_prepare(name, host)
    pilot, f0 = oracle_step_sample(name, host, 1.0 / 64, prepared)
    frac = min(1.0, f0 * target_s / max(pilot, 1e-6))
    t, f = oracle_step_sample(name, host, frac, prepared)
    kind = synth.WORKLOADS[name]["kind"]
    if kind in QUANT_KINDS:
        gbs = quant_step_bytes(synth.WORKLOADS[name], m, k) * f / t / 1e9
        what = {"quant2d": "both directions", "quant_sr": "stochastic rounding",
                "transpose": "FP4 code transpose"}[kind]
        return {"value": gbs, "unit": "GB/s", "cores": oracle_threads(), "kind": "oracle",
                "sample": f"{f:.4f} of one step ({int(round(f * m))} of {m} rows, {what}), "
                          f"{t:.1f} s on the host CPU"}
    value = 2.0 * m * n * k * f / t / 1e12
    return {"value": value, "unit": "TFLOPS", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{f:.5f} of one step ({gemm_block(f, m, n)} with the matching share of "
                      f"the quantize work), {t:.1f} s on the host CPU"}


def gemm_block(f, m, n):
    """The output block a GEMM sample of fraction f covers, in words."""
    g = math.sqrt(f)
    return f"a {int(round(m * g))} x {int(round(n * g))} block of the {m} x {n} output"


# --------------------------------------------------------------------- traffic record

# Source files that define the kernels of each call of the step.
CALL_SOURCES = {
    "gemm": ["gemm.cu", "gemm_pair.cu", "gemm_swap.cu", "mx_device.cuh", "mx_internal.h"],
    "quantize_2d": ["quantize.cu", "mx_device.cuh", "mx_internal.h"],
    "quantize": ["quantize.cu", "mx_device.cuh", "mx_internal.h"],
    "quantize_sr": ["quantize.cu", "mx_device.cuh", "mx_internal.h"],
    "transpose": ["transpose.cu", "mx_device.cuh", "mx_internal.h"],
}


def kernel_source_hash(call):
    """Short hash of the sources of a call's kernels (ties an ncu record to them)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_fp4_bf16_gb300", "csrc")
    for f in sorted(CALL_SOURCES[call]):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name, call):
    """DRAM bytes per call (one launch, or the two of an NVFP4 quantize) from
    the committed ncu summary, if its kernels have not changed since the
    counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path) or call not in CALL_SOURCES:
        return None
    src = kernel_source_hash(call)
    for line in open(path):
        kv = dict(re.findall(r"(\w+)=(\S+)", line))
        if kv.get("workload") == name and kv.get("call") == call and kv.get("source") == src:
            try:
                return float(kv["bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


# --------------------------------------------------------------------- MMA ceiling

def calibrate_all(steps=1 << 16):
    """`--calibrate`: every MMA form and shape, one JSON line each."""
    import torch
    torch.cuda.set_device(0)
    from block_scaled_fp4_bf16_gb300 import build
    build.build()
    import block_scaled_fp4_bf16_gb300 as mx
    names = {mx.MX_MMA_MXF4: "kind::mxf4 scale_vec::2X (UE8M0)",
             mx.MX_MMA_MXF4NVF4_2X: "kind::mxf4nvf4 scale_vec::2X (UE8M0)",
             mx.MX_MMA_MXF4NVF4_4X: "kind::mxf4nvf4 scale_vec::4X (UE4M3)"}
    for pair in (1, 0):
        for form, name in names.items():
            r = mma_ceiling(mx, torch, steps, form=form, pair=pair)
            r["form"] = name + (", cta_group::2, 256x256x64" if pair else ", cta_group::1, 128x256x64")
            print(json.dumps(r), flush=True)


def mma_ceiling(mx, torch, steps=1 << 15, form=None, pair=1):
    """Live calibration of the tensor pipe (mx_calibrate_mma): one wave of
    back-to-back CTA-pair MMAs of the pair GEMM's form and shape per SM pair.
    Returns its FLOPs per clock per SM (cycle counts of every pair, so it does
    not depend on the clock), the TFLOP/s and the clock it ran at."""
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    cyc = torch.zeros(nsm, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream()
    form = mx.MX_MMA_MXF4 if form is None else form
    mx.mx_calibrate_mma(form, pair, 256, cyc)          # warm-up
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    flops, units = mx.mx_calibrate_mma(form, pair, steps, cyc)
    e1.record(stream)
    torch.cuda.synchronize()
    if mx.mx_device_status() != mx.MX_OK:
        return None
    secs = e0.elapsed_time(e1) * 1e-3
    cycles = statistics.median(cyc[:units].cpu().tolist())
    mmas = 4 * steps
    per_sm_flop = 2.0 * 128 * 256 * 64   # one 128x256x64 MMA, or each SM's half of a pair's
    return {"form": "kind::mxf4 block_scale scale_vec::2X, cta_group::2, 256x256x64",
            "cycles_per_mma": cycles / mmas,
            "flop_per_clk_sm": per_sm_flop * mmas / cycles,
            "tflops": flops / secs / 1e12, "mhz": cycles / secs / 1e6, "sms": nsm}


# --------------------------------------------------------------------- main (ours)

def main_ours(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    from block_scaled_fp4_bf16_gb300 import build
    build.build()
    import block_scaled_fp4_bf16_gb300 as mx
    if not mx.mx_available():
        raise SystemExit("libmxfp4 is not usable on this device")

    def barrier():
        if world > 1:
            dist.barrier()

    name = args.workload
    w, m, n, k = workload_shape(name)
    host = synth.workload_inputs(name)
    # rotating input sets: working set > 3x L2
    probe = DeviceWorkload(name, host, 1)
    nsets = max(4, -(-3 * L2_BYTES // probe.set_bytes))
    del probe
    wl = DeviceWorkload(name, host, nsets)
    graphs, stream, ev0, ev1 = time_graphs(wl, args.steps, args.warmup)

    gpu_id = str(local)
    try:
        props = torch.cuda.get_device_properties(local)
        if getattr(props, "uuid", None) is not None:
            gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    time.sleep(0.6)
    # settle clocks under load before the timed region (untimed)
    with torch.cuda.stream(stream):
        t_end = time.time() + 1.0
        while time.time() < t_end:
            graphs[0].replay()
    torch.cuda.synchronize()
    ms, t0, t1 = run_graph_region(wl, graphs, stream, ev0, ev1, args.steps, barrier)
    ms_per_step = reduce_max(ms / args.steps, world, "cuda")

    windows = {}
    per_call = time_calls(wl, args.steps, windows=windows, min_seconds=args.min_call_seconds)
    time.sleep(0.3)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    call_clocks = {c: sampler.summary(*w) for c, w in windows.items()}
    ceiling = mma_ceiling(mx, torch)
    e2e_steps = args.e2e_steps or min(args.steps, 200)
    e2e_ms, h2d, d2h = time_e2e(wl, host, e2e_steps)
    e2e_ms = reduce_max(e2e_ms, world, "cuda")

    peaks, peak_src = load_peaks()
    # every kernel is timed on its own (back-to-back calls of that kernel): the
    # burst bf16 figure is the one that applies, times the nominal FP4 ratio
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    hbm_peak = peaks["hbm_gbs"]
    flops = 2.0 * m * n * k
    quant_only = wl.kind in QUANT_KINDS
    # a quantize-only step has no GEMM: its value is algorithmic GB/s
    step_work = sum(b for b, _ in wl.algorithmic().values()) / 1e9 if quant_only else flops / 1e12
    unit = "GB/s" if quant_only else "TFLOPS"
    value = job_throughput(step_work, ms_per_step, world)
    alg = wl.algorithmic()
    kpc = wl.kernels_per_call()
    kernels = {}
    for label, dur_ms in per_call.items():
        b, f = alg[label]
        t_s = dur_ms * 1e-3
        if f > 0 and f / (fp4_peak * 1e12) >= b / (hbm_peak * 1e9):
            kernels[label] = {"bound": "tensor", "achieved": f / t_s / 1e12, "peak": fp4_peak,
                              "unit": "TFLOP/s", "avg_us": dur_ms * 1e3,
                              "launches_per_step": kpc[label]}
        else:
            kernels[label] = {"bound": "hbm", "achieved": b / t_s / 1e9, "peak": hbm_peak,
                              "unit": "GB/s", "avg_us": dur_ms * 1e3,
                              "launches_per_step": kpc[label]}
        kernels[label]["frac"] = kernels[label]["achieved"] / kernels[label]["peak"]
        kernels[label]["algorithmic_bytes"] = b
        kernels[label]["algorithmic_flops"] = f
        cc = call_clocks.get(label) or {}
        kernels[label]["sm_mhz"] = cc.get("sm_mhz")
        kernels[label]["clock_samples"] = cc.get("samples", 0)
        if f > 0 and ceiling and cc.get("sm_mhz"):
            # FLOPs per clock per SM at the clock the kernel ran at, against the
            # calibrated MMA rate: the tensor-pipe efficiency, independent of
            # the power cap's clock
            fpc = f / t_s / (ceiling["sms"] * cc["sm_mhz"] * 1e6)
            kernels[label]["flop_per_clk_sm"] = fpc
            kernels[label]["frac_of_mma_ceiling_per_clock"] = fpc / ceiling["flop_per_clk_sm"]
    dom = max(per_call, key=lambda c: per_call[c])
    kd = kernels[dom]
    traffic = recorded_traffic(name, dom)
    roofline = {"bound": kd["bound"], "achieved": kd["achieved"], "peak": kd["peak"],
                "unit": kd["unit"], "frac": kd["frac"], "traffic": traffic, "kernel": dom,
                "peak_source": (f"{peak_src} " + ("bf16_tflops (burst) x 6 (nominal FP4:BF16 "
                                                  "dense ratio); the kernel is timed on its own"
                                                  if kd["bound"] == "tensor" else "hbm_gbs"))}
    if kd["bound"] == "tensor":
        roofline["peak_sustained"] = peaks["bf16_tflops_sustained"] * FP4_OVER_BF16
        roofline["frac_of_sustained"] = kd["achieved"] / roofline["peak_sustained"]
        if ceiling:
            roofline["mma_ceiling"] = ceiling
            roofline["sm_mhz"] = kd.get("sm_mhz")
            roofline["frac_of_mma_ceiling_per_clock"] = kd.get("frac_of_mma_ceiling_per_clock")
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("u8 (e2m1 code bytes)" if wl.kind == "transpose" else
                  "bf16 -> e2m1 (quantize only)" if quant_only else "e2m1 (fp32 accumulate)"),
        "data": "synthetic",
        "config": {"workload": name, "m": m, "n": n, "k": k, "format": w["fmt"],
                   "out": w["out"], "rotating_sets": nsets,
                   "l2": f"rotating input sets, {nsets} x {wl.set_bytes / 2**20:.0f} MiB "
                         f"> 3x L2",
                   "parallelism": f"replicas x{world}",
                   "step": " + ".join(per_call.keys())},
        "roofline": roofline,
        "kernels": kernels,
        "sum_of_calls_ms": sum(per_call.values()),
        "e2e": {"value": job_throughput(step_work, e2e_ms, world), "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps * sum(kpc.values()),
        "clocks": clocks,
    }
    if "gemm" in kernels:
        line["gemm_tflops"] = kernels["gemm"]["achieved"] if kernels["gemm"]["unit"] == "TFLOP/s" \
            else flops / (kernels["gemm"]["avg_us"] * 1e-6) / 1e12
        line["gemm_pct_fp4_peak"] = 100.0 * line["gemm_tflops"] / fp4_peak
    qs = [c for c in kernels if c.startswith("quantize")]
    if qs:
        qb = sum(kernels[c]["algorithmic_bytes"] for c in qs)
        qt = sum(kernels[c]["avg_us"] for c in qs) * 1e-6
        line["quantize_gbs"] = qb / qt / 1e9
        line["quantize_pct_hbm"] = 100.0 * line["quantize_gbs"] / hbm_peak
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(name, host, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------------- main (reference)

def main_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    name = args.workload
    _, m, n, k = workload_shape(name)
    host = synth.workload_inputs(name)
    prepared = oracle_prepare(name, host)
    pilot, f0 = oracle_step_sample(name, host, 1.0 / 256, prepared)
    budget = 150.0 / (args.steps + args.warmup)      # seconds per step
    kind = synth.WORKLOADS[name]["kind"]
    smallest = 1.0 / m if kind in QUANT_KINDS else 1.0 / (m * n)   # one row / one output
    frac = min(1.0, max(smallest, f0 * budget / max(pilot, 1e-6)))
    for _ in range(args.warmup):
        oracle_step_sample(name, host, frac, prepared)
    times, f = [], frac
    for _ in range(args.steps):
        t, f = oracle_step_sample(name, host, frac, prepared)
        times.append(t)
    mean_t = statistics.fmean(times)
    quant_only = kind in QUANT_KINDS
    unit = "GB/s" if quant_only else "TFLOPS"
    value = (quant_step_bytes(synth.WORKLOADS[name], m, k) * f / mean_t / 1e9 if quant_only
             else 2.0 * m * n * k * f / mean_t / 1e12)
    sample = (f"{f:.6f} of one step per step ({int(round(f * m))} of {m} rows)" if quant_only
              else f"{f:.6f} of one step per step ({gemm_block(f, m, n)} with the matching "
                   f"share of the quantize work)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": mean_t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": name, "m": m, "n": n, "k": k},
        "cpu_baseline": {"value": value, "unit": unit, "cores": oracle_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse_args()
    if a.calibrate:
        calibrate_all()
    elif a.impl == "reference":
        main_reference(a)
    else:
        main_ours(a)
