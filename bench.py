#!/usr/bin/env python
"""Benchmark of the HLQ/HOT backward pass of one linear layer on GB300.

One step = the whole hot path on one batch of synthetic input:
  ACBP compression of x at forward time (hlq_compress_activation), then the
  backward pass: g_x through int4 Hadamard quantization
  (hlq_linear_backward_gx) and g_w through the Hadamard low-rank
  approximation with int8 (hlq_linear_backward_gw).
Default workload: the largest single-GPU layer of the five, a Llama-3-8B
MLP down_proj: T = 8 x 2048 = 16384 tokens, Cin = 14336, Cout = 4096, bf16
inputs, per-token g_y quantizer.  The other layers (ViT-B qkv and fc2,
ResNet-50 3x3 im2col, the small single linear) are timed the same way in the
line's `per_workload` block.

Prints one JSON line (rank 0).  `value` is microseconds per layer step
(lower is better), device-timed with CUDA events on the launching stream,
inputs resident in HBM, L2 flushed (256 MiB write) before every timed step.
`e2e` is the same step through libhlq's host-buffer entry
(hlq_layer_step_host): pinned host -> device copies of x, g_y, w and
device -> host copies of g_x, g_w inside the timed region, pipelined with the
kernels by the library.
`roofline` is for the kernel with the largest device time, from per-launch
CUDA events recorded by libhlq's tracing hooks.  Algorithmic bytes follow the
method's data sizes, not the library's storage layout: one read of each
input, int4 codes at half a byte, int8 codes at one byte, the scales; a
per-tensor maximum pre-pass re-reads its input and is credited with no bytes;
the GEMMs are credited with their integer operations, their roofline time
being max(ops / tensor peak, (operands + output) / HBM peak).
`cpu_baseline` times the CPU oracle on a bounded sample of the workload on
this host and extrapolates it linearly to the whole layer.

--impl reference times the CPU oracle itself (the only reference there is)
per step on a bounded sample and prints the same metric.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = ("HLQ linear-backward µs/layer & effective TOPS; % of "
          "int8-tensor / HBM roofline")
UNIT = "us/layer"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}
NOMINAL_FP8_OVER_BF16 = 4.5 / 2.25
DEFAULT_WORKLOAD = workloads.WORKLOADS[3]   # Llama-3-8B down_proj: the largest


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD.name,
                   help="workload name or index into workloads.WORKLOADS")
    p.add_argument("--cpu-sample-tokens", type=int, default=256)
    p.add_argument("--cpu-sample-w-rows", type=int, default=512)
    p.add_argument("--ref-sample-tokens", type=int, default=16)
    p.add_argument("--ref-sample-w-rows", type=int, default=64)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-workload", action="store_true",
                   help="time only the main workload")
    p.add_argument("--serial", action="store_true",
                   help="time the g_x and g_w branches one after the other "
                        "instead of concurrently (hlq_linear_backward)")
    p.add_argument("--fused-gy", action="store_true",
                   help="run the step through the fused reader of g_y "
                        "(hlq_linear_backward(fused_gy=True))")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the timings of the optional paths (int4 / "
                        "per-channel ACBP, quantizer selection, ablations)")
    p.add_argument("--profile", choices=["compress", "gx", "gw", "step"],
                   help="no timing: call this one entry point --warmup times on "
                        "the workload and exit (a small, fixed launch sequence "
                        "for a profiler)")
    p.add_argument("--tokens", type=int, default=0,
                   help="with --profile: use the first TOKENS tokens only")
    p.add_argument("--gw-operands", choices=list(GW_MODES), default="auto",
                   help="how the g_w GEMM takes its int8 operands "
                        "(hlq_set_gw_operands): the library's default, x-bar "
                        "widened by its own kernel, x-bar widened in the GEMM's "
                        "shared memory, or both operands kept int8")
    return p.parse_args(argv)


GW_MODES = {"auto": 0, "widen": 1, "int8_x": 2, "int8_both": 3}


def pick_workload(spec):
    if spec.isdigit():
        return workloads.WORKLOADS[int(spec)]
    return workloads.BY_NAME[spec]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


# ----------------------------------------------------------------------------
# algorithmic work per kernel launch and per step of the method
# ----------------------------------------------------------------------------

def _sizes(wl, xbar_bits=8):
    """Bytes of the method's data: element size of the inputs, and the
    code bytes of each quantized tensor (int4 at half a byte, int8 at one)."""
    T, Cin, Cout, Tp = wl.T, wl.Cin, wl.Cout, wl.Tp
    e = 2 if wl.dtype == "bf16" else 4
    per_tok = wl.gran_gy == workloads.PER_TOKEN
    return dict(
        e=e,
        gy=T * Cout * e, x=T * Cin * e, w=Cout * Cin * e,
        qy=T * Cout // 2, s_gy=4 * T if per_tok else 4,       # HQ of g_y: int4
        qw=Cin * Cout // 2, s_w=4,                            # HQ of w: int4
        qg=Cout * Tp, s_g=4,                                  # HLA of g_y: int8
        xb=Cin * Tp if xbar_bits == 8 else Cin * Tp // 2, s_x=4,   # ACBP codes
        gx=T * Cin * 4, gw=Cout * Cin * 4,                    # fp32 outputs
        ops_gx=2 * T * Cin * Cout, ops_gw=2 * Cout * Cin * Tp)


# kernel -> (step of the method it belongs to, how it is credited)
KERNEL_ROWS = {
    "hla_x_amax": "a1", "hla_x_quant": "a1",
    "hq_rows_amax": "a2", "hq_rows_quant": "a2",
    "hq_cols_amax": "a3", "hq_cols_quant": "a3",
    "gemm_gx_tc": "a4",
    "hla_gy_amax": "a5", "hla_gy_quant": "a5",
    "widen_xbar": "a6", "gemm_gw_tc": "a6",
    "gy_fused_amax": "a2+a5", "gy_fused_quant": "a2+a5",
}
ROW_NAMES = {"a1": "ACBP compression of x", "a2": "HQ of g_y", "a3": "HQ of w",
             "a4": "g_x GEMM + dequant", "a5": "HLA of g_y",
             "a6": "g_w GEMM + dequant",
             "a2+a5": "HQ and HLA of g_y by one fused reader (per-tensor g_y scale)"}


def algorithmic(name, wl, xbar_bits=8):
    """What one launch of `name` is credited with: ("hbm", bytes) for the
    transform/quantize kernels, ("ops", integer ops, bytes) for the GEMMs.

    Bytes are the method's: one read of the input plus the codes (int4 at
    0.5 B, int8 at 1 B) and scales written.  The quantize pass of a
    per-tensor quantizer carries them; its maximum pre-pass re-reads the
    input and is credited with nothing, as is the int8 -> bf16 widening of
    the stored activation (a layout step, not one of the method)."""
    s = _sizes(wl, xbar_bits)
    table = {
        "hla_x_amax": ("hbm", 0),
        "hla_x_quant": ("hbm", s["x"] + s["xb"] + s["s_x"]),
        "hq_rows_amax": ("hbm", 0),
        "hq_rows_quant": ("hbm", s["gy"] + s["qy"] + s["s_gy"]),
        "hq_cols_amax": ("hbm", 0),
        "hq_cols_quant": ("hbm", s["w"] + s["qw"] + s["s_w"]),
        "hla_gy_amax": ("hbm", 0),
        "hla_gy_quant": ("hbm", s["gy"] + s["qg"] + s["s_g"]),
        "widen_xbar": ("hbm", 0),
        "gy_fused_amax": ("hbm", 0),
        "gy_fused_quant": ("hbm", s["gy"] + s["qy"] + s["s_gy"] + s["qg"] + s["s_g"]),
        "gemm_gx_tc": ("ops", s["ops_gx"], s["qy"] + s["qw"] + s["gx"]),
        "gemm_gw_tc": ("ops", s["ops_gw"], s["qg"] + s["xb"] + s["gw"]),
    }
    return table.get(name, ("hbm", 0))


ROW_WORK = {  # algorithmic work of each step of the method (same sizes)
    "a1": lambda s: ("hbm", s["x"] + s["xb"] + s["s_x"]),
    "a2": lambda s: ("hbm", s["gy"] + s["qy"] + s["s_gy"]),
    "a3": lambda s: ("hbm", s["w"] + s["qw"] + s["s_w"]),
    "a4": lambda s: ("ops", s["ops_gx"], s["qy"] + s["qw"] + s["gx"]),
    "a5": lambda s: ("hbm", s["gy"] + s["qg"] + s["s_g"]),
    "a6": lambda s: ("ops", s["ops_gw"], s["qg"] + s["xb"] + s["gw"]),
    "a2+a5": lambda s: ("hbm", s["gy"] + s["qy"] + s["s_gy"] + s["qg"] + s["s_g"]),
}


def tensor_peak(name, peaks, sustained=False):
    """Tensor-pipe peak (TFLOP/s) of a GEMM by operand type: E4M3 operands on
    the FP8 pipe (the measured bf16 figure x the nominal FP8/BF16 ratio),
    bf16 operands at the measured bf16 figure."""
    bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    if name.startswith("gemm_gx") or name == "a4":
        return bf16 * NOMINAL_FP8_OVER_BF16
    return bf16


def roofline_of(name, work, seconds, peaks):
    """Achieved rate and fraction of the binding roof for `work` done in
    `seconds`.  A GEMM's roof time is max(ops / tensor peak, bytes / HBM
    peak); the achieved figure is given in the unit of the binding roof."""
    hbm = peaks["hbm_gbs"] * 1e9
    if work[0] == "hbm":
        achieved = work[1] / seconds / 1e9
        return {"bound": "hbm", "achieved": achieved, "unit": "GB/s",
                "peak": peaks["hbm_gbs"], "frac": achieved / peaks["hbm_gbs"],
                "algorithmic": work[1]}
    ops, nbytes = work[1], work[2]
    tp = tensor_peak(name, peaks) * 1e12
    if ops / tp >= nbytes / hbm:
        achieved = ops / seconds / 1e12
        return {"bound": "tensor", "achieved": achieved, "unit": "TFLOP/s",
                "peak": tp / 1e12, "frac": achieved / (tp / 1e12),
                "algorithmic": ops, "bytes": nbytes}
    achieved = nbytes / seconds / 1e9
    return {"bound": "hbm", "achieved": achieved, "unit": "GB/s",
            "peak": peaks["hbm_gbs"], "frac": achieved / peaks["hbm_gbs"],
            "algorithmic": nbytes, "ops": ops}


def kernel_table(launches, wl, peaks, xbar_bits=8):
    """Per-kernel and per-step summaries of traced launches [(name, ms)]."""
    per_kernel = {}
    for name, kms in launches:
        d = per_kernel.setdefault(name, [0, 0.0])
        d[0] += 1
        d[1] += kms
    total = sum(v[1] for v in per_kernel.values()) or 1.0
    kernels = {}
    for name, (n, tot) in sorted(per_kernel.items(), key=lambda kv: -kv[1][1]):
        avg_s = tot / n / 1e3
        entry = {"launches": n, "avg_us": avg_s * 1e6, "share": tot / total,
                 "row": KERNEL_ROWS.get(name)}
        work = algorithmic(name, wl, xbar_bits)
        if work[1] > 0:
            entry.update(roofline_of(name, work, avg_s, peaks))
        else:
            entry.update({"bound": "hbm", "achieved": 0.0, "frac": 0.0,
                          "note": ("a re-read or layout pass: the method's bytes are "
                                   "credited to the step's other pass")})
        kernels[name] = entry
    s = _sizes(wl, xbar_bits)
    rows = {}
    for row, fn in ROW_WORK.items():
        names = [k for k, r in KERNEL_ROWS.items() if r == row and k in kernels]
        if not names:
            continue
        us = sum(kernels[k]["avg_us"] for k in names)
        r = roofline_of(row, fn(s), us / 1e6, peaks)
        r.update({"what": ROW_NAMES[row], "us": us, "kernels": names})
        rows[row] = r
    return kernels, rows


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="hlq_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU oracle timing (test infrastructure: only this leg runs it)
# ----------------------------------------------------------------------------

def oracle_layer_seconds(wl, inp, tokens, w_rows=None):
    """Oracle time of one layer step split into its two parts, in seconds:
    the HQ of w on its first `w_rows` rows (whole 16-row blocks; all rows by
    default), and everything that grows with the token count (compression
    of x, HQ and HLA of g_y, both integer GEMMs, the dequantizations) on the
    first `tokens` tokens.  Each part is linear in its sample size."""
    import oracle
    oracle.build()
    Ts = tokens
    rows = wl.Cout if w_rows is None else max(16, min(wl.Cout, w_rows // 16 * 16))
    gy = inp["g_y"][:Ts]
    x = inp["x"][:Ts]
    t0 = time.perf_counter()
    Wt = oracle.hq_transform(inp["w"][:rows], 1)
    qWt, s_w = oracle.hq_quantize(Wt, oracle.PER_TENSOR, oracle.SR, wl.seed,
                                  oracle.STREAM_W)
    t_w = time.perf_counter() - t0
    # the g_x GEMM contracts over all Cout: the sampled rows of w stand in
    # for every block (timing only; the codes are not compared here)
    reps = wl.Cout // rows
    qW = np.ascontiguousarray(np.tile(qWt, (reps, 1)).T)
    t1 = time.perf_counter()
    qx, s_x = oracle.compress_activation(x, wl.rank)
    Y = oracle.hq_transform(gy, 0)
    qY, s_gy = oracle.hq_quantize(Y, wl.gran_gy, oracle.SR, wl.seed,
                                  oracle.STREAM_GY)
    acc = oracle.gemm_i64(qY, qW)
    oracle.dequant_gx(acc, s_gy, wl.gran_gy, s_w[0])
    oracle.gw_path(gy, qx, s_x, wl.rank)
    t_tok = time.perf_counter() - t1
    return t_w * (wl.Cout / rows), t_tok, rows


def host_cpu(cpuinfo="/proc/cpuinfo"):
    """The host the oracle runs on: machine, logical CPUs, and the CPU model
    where /proc/cpuinfo names one (Arm hosts give implementer and part
    codes instead).  Never raises."""
    info = {"machine": platform.machine(), "nproc": os.cpu_count(), "model": None}
    try:
        fields = {}
        with open(cpuinfo) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
        if fields.get("model name"):
            info["model"] = fields["model name"]
        elif fields.get("cpu implementer") or fields.get("cpu part"):
            info["model"] = (f"implementer {fields.get('cpu implementer')} "
                             f"part {fields.get('cpu part')}")
    except (OSError, UnicodeDecodeError):
        pass
    return info


def _sample_text(wl, tokens, rows, t_tok=None, t_w=None):
    tok = f" ({t_tok:.2f} s)" if t_tok is not None else ""
    wpart = (f"the HQ of w on {rows} of {wl.Cout} rows"
             + (f" ({t_w * rows / wl.Cout:.2f} s)" if t_w is not None else "")
             + (f" scaled by Cout/{rows}" if rows < wl.Cout else ""))
    return (f"oracle on the first {tokens} of {wl.T} tokens{tok} (compression, "
            f"HQ and HLA of g_y, both integer GEMMs) scaled by T/{tokens}, plus "
            f"{wpart}; single thread; extrapolated linearly")


def cpu_baseline(wl, inp, tokens, w_rows=None):
    t_w, t_tok, rows = oracle_layer_seconds(wl, inp, tokens, w_rows)
    est = t_w + t_tok * (wl.T / tokens)
    return {"value": est * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": _sample_text(wl, tokens, rows, t_tok, t_w),
            "extrapolated": tokens < wl.T or rows < wl.Cout,
            "measured_s": t_w * rows / wl.Cout + t_tok, "host": host_cpu()}


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------

def run_reference(args, wl, rank, world):
    if rank != 0:
        return 0
    tokens = max(16, args.ref_sample_tokens // 16 * 16)
    inp = workloads.make_inputs(wl, T=tokens)
    per_step = []
    rows = wl.Cout
    for i in range(args.warmup + args.steps):
        t_w, t_tok, rows = oracle_layer_seconds(wl, inp, tokens, args.ref_sample_w_rows)
        if i >= args.warmup:
            per_step.append(t_w + t_tok * (wl.T / tokens))
    us = statistics.mean(per_step) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "per step: " + _sample_text(wl, tokens, rows),
                         "extrapolated": True, "host": host_cpu()},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks(value, dist=None, device="cpu"):
    """The largest of every rank's value (the job is as slow as its slowest
    replica); the value itself without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_layer(ms_per_step, world):
    """Job-wide microseconds per layer step: `world` replicas each finish one
    step in `ms_per_step` (weak scaling)."""
    return ms_per_step * 1e3 / world


def config_of(wl):
    return {"workload": wl.name, "T": wl.T, "Cin": wl.Cin, "Cout": wl.Cout,
            "input_dtype": wl.dtype, "block": wl.block, "rank": wl.rank,
            "gran_gy": "per-token" if wl.gran_gy else "per-tensor",
            "branches": "serial" if getattr(ARGS, "serial", False) else "overlapped",
            "gy_reader": "fused" if getattr(ARGS, "fused_gy", False) else "separate",
            "entry": ("hlq_compress_activation + hlq_linear_backward"
                      if getattr(ARGS, "serial", False) or getattr(ARGS, "fused_gy", False)
                      else "hlq_layer_step (compression beside the g_x branch)"),
            "gw_operands": getattr(ARGS, "gw_operands", "auto"),
            "l2": "flushed before every timed step (256 MiB write)"}


def measure_workload(args, wl, dev, dist, headline):
    """Device-timed step of one workload, its backward and compression alone,
    and the per-kernel attribution; for the headline workload also the
    optional paths, the end-to-end host-buffer step and the clocks."""
    import torch
    import hadamard_precision_backprop_gb300 as hlq

    def barrier():
        if dist is not None:
            dist.barrier()

    inp = workloads.make_inputs(wl)
    e = 2 if wl.dtype == "bf16" else 4

    def host_tensor(name):
        if wl.dtype == "bf16":
            t = torch.from_numpy(inp[name + "_bits"].view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(inp[name])
        return t.pin_memory()

    h_x, h_gy, h_w = host_tensor("x"), host_tensor("g_y"), host_tensor("w")
    x, gy, w = (t.to(dev) for t in (h_x, h_gy, h_w))
    T, Cin, Cout, Tp = wl.T, wl.Cin, wl.Cout, wl.Tp
    ws0 = hlq.workspace(hlq.OP_COMPRESS_ACTIVATION, T, Cin, Cout, 16, wl.rank, dev)
    ws1 = hlq.workspace(hlq.OP_BACKWARD_FUSED, T, Cin, Cout, 16, wl.rank, dev)
    ws_step = hlq.workspace(hlq.OP_LAYER_STEP, T, Cin, Cout, 16, wl.rank, dev)
    xbar = torch.empty((Cin, Tp), dtype=torch.int8, device=dev)
    sx = torch.empty(1, dtype=torch.float32, device=dev)
    gx = torch.empty((T, Cin), dtype=torch.float32, device=dev)
    gw = torch.empty((Cout, Cin), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(xx, gg, ww, overlap=None):
        # forward-time ACBP, then both gradients
        overlap = (not args.serial) if overlap is None else overlap
        if overlap and not args.fused_gy:
            # one call: the compression runs on the g_w branch, beside the
            # g_x branch (hlq_layer_step)
            hlq.hlq_layer_step(xx, gg, ww, rank=wl.rank, gran_gy=wl.gran_gy,
                               gran_w=wl.gran_w, rnd=hlq.SR, seed=wl.seed, out_gx=gx,
                               out_gw=gw, xbar=xbar, xbar_scale=sx, ws=ws_step)
            return
        hlq.hlq_compress_activation(xx, rank=wl.rank, out=xbar, scale=sx, ws=ws0)
        if overlap or args.fused_gy:   # g_w branch on a second stream inside the library
            hlq.hlq_linear_backward(gg, ww, xbar, sx, rank=wl.rank,
                                    gran_gy=wl.gran_gy, gran_w=wl.gran_w,
                                    rnd=hlq.SR, seed=wl.seed, out_gx=gx,
                                    out_gw=gw, ws=ws1, fused_gy=args.fused_gy)
        else:
            hlq.hlq_linear_backward_gx(gg, ww, gran_gy=wl.gran_gy, gran_w=wl.gran_w,
                                       rnd=hlq.SR, seed=wl.seed, out=gx, ws=ws1)
            hlq.hlq_linear_backward_gw(gg, xbar, sx, rank=wl.rank, out=gw, ws=ws1)

    def traced_step():
        # the step's own call with every branch on this stream in turn
        hlq.hlq_debug_serialize_branches(True)
        try:
            step(x, gy, w)
        finally:
            hlq.hlq_debug_serialize_branches(False)

    # ---- device-resident timing ------------------------------------------
    # The step is captured into a CUDA graph and replayed (no host launch
    # gaps).  Timed region: each step = L2 flush (outside the events), then
    # one replay between two events.  Per-kernel attribution comes from a
    # second graph of the same step whose launches are bracketed by libhlq's
    # trace events (event boundaries serialise neighbouring kernels, so
    # those per-kernel times are slightly pessimistic); it is replayed right
    # after the timed region, one traced step per timed step.
    for _ in range(args.warmup):
        step(x, gy, w)
    torch.cuda.synchronize()
    graph = traced = None
    timing = "CUDA graph replay of the step"
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(x, gy, w)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(x, gy, w)
        # per-kernel attribution: the same call with its branches one after
        # the other, so each kernel's traced time is its own (as in a
        # serialised profiler run)
        traced = torch.cuda.CUDAGraph()
        hlq.hlq_trace_begin(256)
        with torch.cuda.graph(traced):
            traced_step()
        hlq.hlq_trace_end(keep=True)
        for _ in range(args.warmup):
            graph.replay()
            traced.replay()
    except Exception as exc:  # capture unsupported: eager steps, traced live
        graph = traced = None
        timing = f"eager launches (graph capture failed: {type(exc).__name__})"
        hlq.hlq_trace_free()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        flush.fill_(1)
        a.record(stream)
        if graph is not None:
            graph.replay()
        else:
            step(x, gy, w)
        b.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms = statistics.mean(step_ms)
    ms = max_over_ranks(ms, dist, dev)
    launches = []
    for _ in range(args.steps):
        flush.fill_(1)
        if traced is not None:
            traced.replay()
            torch.cuda.synchronize()
            launches += hlq.hlq_trace_read()
        else:
            hlq.hlq_trace_begin(256)
            traced_step()
            torch.cuda.synchronize()
            launches += hlq.hlq_trace_end()
    if traced is not None:
        hlq.hlq_trace_free()
    del graph, traced

    # ---- the optional paths, each timed alone on the same inputs ----------
    # (graph replay, L2 flushed before each replay, mean over the steps)
    def time_replays(fn):
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        for _ in range(args.warmup):
            g.replay()
        ts = []
        for _ in range(args.steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ts) * 1e3

    # the backward alone (rows a2-a7: both gradients from the stored
    # activation) and the forward-time compression alone, each its own graph
    def backward_only():
        hlq.hlq_linear_backward(gy, w, xbar, sx, rank=wl.rank, gran_gy=wl.gran_gy,
                                gran_w=wl.gran_w, rnd=hlq.SR, seed=wl.seed, out_gx=gx,
                                out_gw=gw, ws=ws1)

    def forward_only():
        hlq.hlq_compress_activation(x, rank=wl.rank, out=xbar, scale=sx, ws=ws0)

    bwd_us = time_replays(backward_only)
    fwd_us = time_replays(forward_only)
    peaks = load_peaks()
    kernels, rows = kernel_table(launches, wl, peaks)
    top = next(iter(kernels))
    roofline = {k: kernels[top][k] for k in ("bound", "achieved", "peak", "unit", "frac")
                if k in kernels[top]}
    roofline.update({"kernel": top, "traffic": load_traffic(top, wl),
                     "peak_source": peaks["source"]})
    if "peak" not in roofline:
        roofline["peak"] = peaks["hbm_gbs"]
    gemm_s = sum(v["avg_us"] * v["launches"] for k, v in kernels.items()
                 if k.startswith("gemm")) / args.steps / 1e6
    gemm_ops = 2 * T * Cin * Cout + 2 * Cout * Cin * Tp
    gemm_bitops = 2 * T * Cin * Cout * 4 + 2 * Cout * Cin * Tp * 8
    res = {
        "ms_per_step": ms,
        "us_per_layer": ms * 1e3,
        # each timed alone (graph replays, L2 flushed): the backward from the
        # stored activation, and the forward-time compression; the step
        # overlaps the compression with the g_x branch
        "backward_us": bwd_us,
        "forward_acbp_us": fwd_us,
        # vanilla-equivalent work of the backward (two dense GEMMs of
        # 2*T*Cin*Cout each) per second of the measured backward
        "effective_tops": 4 * T * Cin * Cout / (bwd_us / 1e6) / 1e12,
        # integer ops the two GEMMs execute (reduced K = T' on the g_w side),
        # per second of their traced time; and those ops x operand bits
        "gemm_int_tops": gemm_ops / gemm_s / 1e12 if gemm_s > 0 else None,
        "gemm_tbops": gemm_bitops / gemm_s / 1e12 if gemm_s > 0 else None,
        "roofline": roofline,
        "kernels": kernels,
        "rows": rows,
        "gpu_launches": len(launches),
        "timing": timing,
        "clocks": clk,
        "config": config_of(wl),
    }
    variants = {}
    if headline and not args.no_variants and (dist is None):
        xb4 = torch.empty(hlq.xbar_shape(T, Cin, wl.rank, 4), dtype=torch.uint8, device=dev)
        sxc = torch.empty(Cin, dtype=torch.float32, device=dev)
        mse = torch.empty(2, dtype=torch.float64, device=dev)
        choice = torch.empty(1, dtype=torch.int32, device=dev)
        ws_sel = hlq.workspace(hlq.OP_SELECT_GRANULARITY, T, Cin, Cout, 16, 8, dev)
        ws_agw = hlq.workspace(hlq.OP_ABLATION_GW_HQ, T, Cin, Cout, 16, 8, dev)
        ws_agx = hlq.workspace(hlq.OP_ABLATION_GX_HLA, T, Cin, Cout, 16, wl.rank, dev)
        gw_a = torch.empty((Cout, Cin), dtype=torch.float32, device=dev)
        gx_a = torch.empty((T, Cin), dtype=torch.float32, device=dev)

        def step_int4():
            hlq.hlq_compress_activation(x, rank=wl.rank, out=xb4, scale=sx, ws=ws0,
                                        xbar_bits=4)
            hlq.hlq_linear_backward(gy, w, xb4, sx, rank=wl.rank, gran_gy=wl.gran_gy,
                                    gran_w=wl.gran_w, rnd=hlq.SR, seed=wl.seed,
                                    out_gx=gx, out_gw=gw, ws=ws1, xbar_bits=4)

        def step_per_channel():
            hlq.hlq_compress_activation(x, rank=wl.rank, out=xbar, scale=sxc, ws=ws0,
                                        xbar_per_channel=True)
            hlq.hlq_linear_backward(gy, w, xbar, sxc, rank=wl.rank, gran_gy=wl.gran_gy,
                                    gran_w=wl.gran_w, rnd=hlq.SR, seed=wl.seed,
                                    out_gx=gx, out_gw=gw, ws=ws1, xbar_per_channel=True)

        def step_fused_gy():
            hlq.hlq_compress_activation(x, rank=wl.rank, out=xbar, scale=sx, ws=ws0)
            hlq.hlq_linear_backward(gy, w, xbar, sx, rank=wl.rank, gran_gy=wl.gran_gy,
                                    gran_w=wl.gran_w, rnd=hlq.SR, seed=wl.seed,
                                    out_gx=gx, out_gw=gw, ws=ws1, fused_gy=True)

        def select():
            hlq.hlq_select_gy_granularity(gy, mse=mse, choice=choice, ws=ws_sel)

        def ablation_gw():
            hlq.hlq_ablation_gw_hq(gy, x, rnd=hlq.SR, seed=wl.seed, out=gw_a, ws=ws_agw)

        def ablation_gx():
            hlq.hlq_ablation_gx_hla(gy, w, rank=wl.rank, out=gx_a, ws=ws_agx)

        def step_gw_mode(mode):
            def fn():
                prev = hlq.hlq_get_gw_operands()
                hlq.hlq_set_gw_operands(mode)
                try:
                    step(x, gy, w)
                finally:
                    hlq.hlq_set_gw_operands(prev)
            return fn

        for name, fn, what in [
                ("fused_gy_step", step_fused_gy,
                 "whole step with one fused reader of g_y for HQ and HLA"),
                ("acbp_int4_step", step_int4,
                 "whole step with the stored activation as packed int4 codes"),
                ("acbp_per_channel_step", step_per_channel,
                 "whole step with one scale per input channel of the stored activation"),
                ("select_gy_granularity", select,
                 "per-token vs per-tensor choice from the int4 RNE MSE of g_y"),
                ("ablation_gw_hq", ablation_gw,
                 "g_w through HQ along tokens and an int4 GEMM over T"),
                ("ablation_gx_hla", ablation_gx,
                 "g_x through HLA along Cout and an int8 GEMM over Cout*rank/16"),
                ("gw_widen_step", step_gw_mode(hlq.GW_WIDEN),
                 "whole step, x-bar widened to fp16 by its own kernel"),
                ("gw_int8_x_step", step_gw_mode(hlq.GW_INT8_X),
                 "whole step, the g_w GEMM widening int8 x-bar in shared memory"),
                ("gw_int8_both_step", step_gw_mode(hlq.GW_INT8_BOTH),
                 "whole step, both g_w operands int8 in HBM, widened in shared memory")]:
            try:
                variants[name] = {"us": time_replays(fn), "what": what}
            except Exception as exc:  # report, do not fail the main line
                variants[name] = {"us": None, "error": f"{type(exc).__name__}: {exc}"}
        torch.cuda.synchronize()
        del xb4, sxc, ws_sel, ws_agw, ws_agx, gw_a, gx_a
        torch.cuda.empty_cache()
    res["variants"] = variants

    # ---- end to end through host buffers ---------------------------------
    # libhlq's host-buffer entry: pinned inputs in, gradients back out, the
    # copies pipelined with the kernels inside the call
    h_gx = torch.empty((T, Cin), dtype=torch.float32).pin_memory()
    h_gw = torch.empty((Cout, Cin), dtype=torch.float32).pin_memory()
    dt_code = hlq.BF16 if wl.dtype == "bf16" else hlq.F32
    ws_host = torch.empty(max(hlq.hlq_layer_step_host_workspace_bytes(
        dt_code, T, Cin, Cout, 16, wl.rank), 256), dtype=torch.uint8, device=dev)

    def e2e_step():
        hlq.hlq_layer_step_host(h_x, h_gy, h_w, xbar, sx, rank=wl.rank,
                                gran_gy=wl.gran_gy, gran_w=wl.gran_w, rnd=hlq.SR,
                                seed=wl.seed, out_gx=h_gx, out_gw=h_gw, ws=ws_host)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e2e_ms, enqueue_ms = [], []
    # the host enqueues every step inside the timed region, so a collection
    # pause of the interpreter would be timed as GPU idle: none during it
    gc.collect()
    gc.disable()
    for _ in range(args.steps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h0 = time.perf_counter()
        e2e_step()
        enqueue_ms.append((time.perf_counter() - h0) * 1e3)
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    gc.enable()
    # the median step: the copies share the host's memory with other jobs on
    # the machine, and single steps have taken 10x longer with the host idle
    # (its enqueue time unchanged); the mean is reported beside it
    e2e = statistics.median(e2e_ms)
    e2e = max_over_ranks(e2e, dist, dev)
    barrier()
    res["e2e_ms"] = e2e
    res["e2e_spread"] = {"statistic": "median of the timed steps",
                         "mean_us": statistics.mean(e2e_ms) * 1e3,
                         "min_us": min(e2e_ms) * 1e3, "median_us": statistics.median(e2e_ms) * 1e3,
                         "max_us": max(e2e_ms) * 1e3,
                         "host_enqueue_us": statistics.median(enqueue_ms) * 1e3,
                         "host_enqueue_max_us": max(enqueue_ms) * 1e3,
                         "steps_us": [round(t * 1e3, 1) for t in e2e_ms]}
    # the copies alone, the floor of that step: the same bytes with plain
    # pinned-memory copies, host -> device and device -> host on two streams
    # at once (the inputs are overwritten with their own values)
    cin_s, cout_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def copies_only():
        cin_s.wait_stream(stream)
        cout_s.wait_stream(stream)
        with torch.cuda.stream(cin_s):
            for d, h in ((w, h_w), (gy, h_gy), (x, h_x)):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(cout_s):
            h_gx.copy_(gx, non_blocking=True)
            h_gw.copy_(gw, non_blocking=True)
        stream.wait_stream(cin_s)
        stream.wait_stream(cout_s)

    floor_ms = []
    for i in range(2 + 5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copies_only()
        b.record(stream)
        b.synchronize()
        if i >= 2:
            floor_ms.append(a.elapsed_time(b))
    res["e2e_spread"]["copy_floor_us"] = statistics.median(floor_ms) * 1e3
    res["e2e_bytes"] = ((x.numel() + gy.numel() + w.numel()) * e,
                        (gx.numel() + gw.numel()) * 4)
    res["acbp_stored_bytes"] = acbp_bytes(T, Cin, wl.rank, e)
    if not headline:
        del x, gy, w, ws0, ws1, ws_step, xbar, gx, gw, flush, ws_host, h_gx, h_gw
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res, inp


def run_profile(args, wl):
    """Call one entry point of the step on the workload's inputs (optionally
    its first --tokens tokens), --warmup times, and return: what a profiler
    captures, with no timing of its own."""
    import dataclasses
    import torch
    import hadamard_precision_backprop_gb300 as hlq
    from hadamard_precision_backprop_gb300 import build as hbuild

    hbuild.build()
    hlq.lib()
    hlq.hlq_set_gw_operands(GW_MODES[args.gw_operands])
    if args.tokens:
        wl = dataclasses.replace(wl, T=min(wl.T, args.tokens // 16 * 16))
    inp = workloads.make_inputs(wl, T=wl.T)
    torch.cuda.set_device(0)

    def dev(name):
        if wl.dtype == "bf16":
            return torch.from_numpy(inp[name + "_bits"].view(np.int16)).view(
                torch.bfloat16).cuda()
        return torch.from_numpy(inp[name]).cuda()

    x, gy, w = dev("x"), dev("g_y"), dev("w")
    xbar, sx = hlq.hlq_compress_activation(x, rank=wl.rank)
    torch.cuda.synchronize()
    for _ in range(max(1, args.warmup)):
        if args.profile == "compress":
            hlq.hlq_compress_activation(x, rank=wl.rank, out=xbar, scale=sx)
        elif args.profile == "gx":
            hlq.hlq_linear_backward_gx(gy, w, gran_gy=wl.gran_gy, gran_w=wl.gran_w,
                                       rnd=hlq.SR, seed=wl.seed)
        elif args.profile == "gw":
            hlq.hlq_linear_backward_gw(gy, xbar, sx, rank=wl.rank)
        else:
            hlq.hlq_layer_step(x, gy, w, rank=wl.rank, gran_gy=wl.gran_gy,
                               gran_w=wl.gran_w, rnd=hlq.SR, seed=wl.seed,
                               xbar=xbar, xbar_scale=sx)
    torch.cuda.synchronize()
    print(json.dumps({"profiled": args.profile, "workload": wl.name, "T": wl.T,
                      "calls": max(1, args.warmup)}))
    return 0


def run_ours(args, wl, rank, world, local_rank):
    import torch
    import hadamard_precision_backprop_gb300 as hlq
    from hadamard_precision_backprop_gb300 import build as hbuild

    hbuild.build()
    hlq.lib()
    hlq.hlq_set_gw_operands(GW_MODES[args.gw_operands])
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

    res, inp = measure_workload(args, wl, dev, dist, headline=True)
    per_workload = {}
    if not args.no_per_workload:
        for other in workloads.WORKLOADS:
            if other.name == wl.name:
                continue
            r, _ = measure_workload(args, other, dev, dist, headline=False)
            entry = {k: r[k] for k in ("us_per_layer", "backward_us", "forward_acbp_us",
                                       "effective_tops", "gemm_int_tops", "roofline",
                                       "rows", "kernels", "clocks")}
            entry["e2e"] = {"value": r["e2e_ms"] * 1e3, "unit": UNIT,
                            "h2d_bytes_per_step": r["e2e_bytes"][0],
                            "d2h_bytes_per_step": r["e2e_bytes"][1], **r["e2e_spread"]}
            per_workload[other.name] = entry
    if rank != 0:
        return 0

    us = job_us_per_layer(res["ms_per_step"], world)      # job-wide us per layer step
    line = {
        "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4/int8", "data": "synthetic",
        "config": res["config"],
        "backward_us": res["backward_us"],
        "forward_acbp_us": res["forward_acbp_us"],
        "effective_tops": res["effective_tops"],
        "gemm_int_tops": res["gemm_int_tops"],
        "gemm_tbops": res["gemm_tbops"],
        "acbp_stored_bytes": res["acbp_stored_bytes"],
        "timing": res["timing"],
        "roofline": res["roofline"],
        "rows": res["rows"],
        "kernels": res["kernels"],
        "gpu_launches": res["gpu_launches"],
        "variants": res["variants"],
        "clocks": res["clocks"],
        "e2e": {"value": job_us_per_layer(res["e2e_ms"], world), "unit": UNIT,
                "h2d_bytes_per_step": res["e2e_bytes"][0],
                "d2h_bytes_per_step": res["e2e_bytes"][1], **res["e2e_spread"]},
        "per_workload": per_workload,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp, min(args.cpu_sample_tokens, wl.T),
                                            args.cpu_sample_w_rows)
    print(json.dumps(line), flush=True)
    return 0


def kernel_sources_digest():
    """sha256 over the CUDA sources that hold device code (kernels, device
    functions and their launch configurations), so that DRAM counters taken
    from an older build of the kernels are not reported against the current
    ones.  Host-only files (the C ABI layer) do not enter it."""
    import hashlib
    d = os.path.join(ROOT, "hadamard_precision_backprop_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(d, name), "rb") as f:
                src = f.read()
            if b"__global__" not in src and b"__device__" not in src:
                continue
            h.update(name.encode())
            h.update(src)
    return h.hexdigest()


def acbp_bytes(T, Cin, rank, e):
    """Bytes of the activation kept for the backward pass: x itself, or the
    ACBP buffer with int8 or packed int4 codes (plus its 4-byte scale)."""
    Tp = T // 16 * rank
    raw = T * Cin * e
    i8 = Cin * Tp + 4
    i4 = Cin * Tp // 2 + 4
    return {"x": raw, "int8": i8, "int4": i4,
            "saved_int8": 1 - i8 / raw, "saved_int4": 1 - i4 / raw}


def load_traffic(kernel, wl):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    capture summary, or None when there is no capture of this kernel on this
    workload or the kernel sources changed after it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("sources_sha256") != kernel_sources_digest():
        return None
    v = d.get("workloads", {}).get(wl.name, {}).get(kernel)
    return None if v is None else v.get("dram_bytes_per_launch")


ARGS = None


def main():
    global ARGS
    args = parse_args()
    ARGS = args
    wl = pick_workload(args.workload)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, wl, rank, world)
    if args.profile:
        return run_profile(args, wl)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        return run_ours(args, wl, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
