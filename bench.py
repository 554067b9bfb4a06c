#!/usr/bin/env python
"""Attention forward+backward throughput on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
attn_fwd (out, lse) then attn_bwd (Delta preprocess, main backward with
atomic dQ partials, dQ convert) through the library's C ABI.

Default workload: the long-sequence configuration at its largest size,
B=1, H=16, S=131072, D=128, bf16, non-causal; q, k, v, dO ~ N(0,1) (seeded).
Every input tensor (512 MiB each) is far larger than the 129 MB L2, so no L2
flush is needed between steps.

Metric: fwd+bwd TFLOP/s with algorithmic flops 3.5 * 4*B*H*S^2*D (halved when
causal).  Prints ONE JSON line (rank 0).  `--impl reference` times the fp64
CPU oracle instead (a bounded sample of the same workload).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOP/s (% of GB300 bf16 tensor peak; non-finite count = 0)"
KERNEL_SOURCES = ("softmax_attention_numerics_gb300/csrc/bwd_sm100.cu",
                  "softmax_attention_numerics_gb300/csrc/sm100_ptx.cuh",
                  "softmax_attention_numerics_gb300/csrc/device_common.cuh")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seqlen", type=int, default=131072)
    ap.add_argument("--heads", type=int, default=16)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--head-dim", type=int, default=128, choices=[64, 128])
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f16", "e4m3"],
                    help="element type of q, k, v, dO and of the outputs; e4m3: the fp8 "
                         "forward alone (bf16 out)")
    ap.add_argument("--deterministic", action="store_true",
                    help="dQ by the per-query-tile kernel instead of fp32 reductions")
    ap.add_argument("--workload", default="attention", choices=["attention", "score", "sparse"],
                    help="score: the head-summed score recompute; sparse: the sparse top-k "
                         "backward with a sink (each its own metric and line)")
    ap.add_argument("--sparse-dim", type=int, default=576, choices=[512, 576],
                    help="kv row width of the sparse workload (576: values in the first 512)")
    ap.add_argument("--topk", type=int, default=128, help="index entries per token (sparse)")
    ap.add_argument("--sparse-batch", type=int, default=16,
                    help="sequences of 512 queries over 2048 kv rows (sparse)")
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="kv heads of the score workload (0: 1, all q heads share it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-oracle-sample", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-oracle-reps", type=int, default=1, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def fwd_flops(B, H, S, D, causal):
    f = 4.0 * B * H * S * S * D
    return f / 2 if causal else f


def workload_name(a):
    return "long_seq B=1 H=%d S=%d D=%d %s%s fwd+bwd%s" % (
        a.heads, a.seqlen, getattr(a, "head_dim", 128), "causal" if a.causal else "non-causal",
        " fp16" if getattr(a, "dtype", "bf16") == "f16" else "",
        " (deterministic dQ)" if a.deterministic else "")


# ---------------------------------------------------------------- CPU oracle sample

def oracle_sample_rows(S):
    """Query rows of head 0 used as the bounded CPU sample (about 8 s of fp64
    arithmetic per repetition on 16 Grace cores at S = 131072)."""
    return max(64, min(S, int(4096 * (131072 / S))))


def run_oracle_sample(a):
    """Child process: time the fp64 oracle on query rows [0, m) of head 0
    against all S keys (full forward+backward arithmetic of those rows)."""
    import numpy as np
    from oracle import attn_oracle as O
    S, D, m = a.seqlen, a.head_dim, a.cpu_oracle_sample
    rng = np.random.default_rng(42)
    q = rng.standard_normal((m, D)).astype(np.float32).astype(np.float64)
    k = rng.standard_normal((S, D)).astype(np.float32).astype(np.float64)
    v = rng.standard_normal((S, D)).astype(np.float32).astype(np.float64)
    do = rng.standard_normal((m, D)).astype(np.float32).astype(np.float64)
    blk = 512                      # rows per oracle call: bounds the host memory
    starts = list(range(0, m, blk))
    zeros = None if a.causal else np.zeros((min(m, blk), S))   # non-causal: no bias at all
    times = []
    vis = 0.0
    for rep in range(a.cpu_oracle_reps):
        t0 = time.perf_counter()
        for r0 in starts:
            r1 = min(m, r0 + blk)
            if a.causal:
                bias = O.bias_for(None, 0, 0, S, S, True, rows=np.arange(r0, r1))
            else:
                bias = zeros[: r1 - r0]
            P, out, lse = O._fwd_head(q[r0:r1], k, v, bias, 1.0 / math.sqrt(D))
            O._bwd_head(q[r0:r1], k, v, P, do[r0:r1], 1.0 / math.sqrt(D))
            if rep == 0:
                vis += float(np.isfinite(bias).sum())
            del P, bias
        times.append(time.perf_counter() - t0)
    flops = 3.5 * 4.0 * vis * D
    print(json.dumps({"times": times, "flops": flops, "rows": m}))


def cpu_oracle(a, rows, reps):
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(cores)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-oracle-sample", str(rows),
           "--cpu-oracle-reps", str(reps), "--seqlen", str(a.seqlen),
           "--head-dim", str(a.head_dim)]
    if a.causal:
        cmd.append("--causal")
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    res["cores"] = cores
    return res


def cpu_baseline_entry(a, res):
    t = min(res["times"])
    return {"value": res["flops"] / t / 1e12, "unit": "TFLOP/s", "cores": res["cores"],
            "kind": "oracle",
            "sample": "fp64 numpy oracle, full fwd+bwd arithmetic of query rows 0..%d of one head "
                      "against all %d keys (%.3g flop in %.2f s)" % (res["rows"] - 1, a.seqlen,
                                                                   res["flops"], t)}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- helpers

# Nominal dense bf16 tensor-core peak of one GB300 (the target is stated against it).
NOMINAL_BF16_TFLOPS = 2250.0


def measured_peaks():
    """The machine's measured peaks, or the fallback figures, said so on stderr
    and in every roofline entry ("peak_source")."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        print("bench.py: %s is missing or unreadable; roofline fractions below are against the "
              "FALLBACK peaks (6.8 TB/s, 1.9 / 1.7 PFLOP/s bf16)" % p, file=sys.stderr)
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def peak_fractions(value, peaks, kind):
    """value (TFLOP/s) against every bf16 denominator: the nominal dense peak
    (the one the 60 % target names), the burst and the sustained peak."""
    burst = peaks.get("bf16_tflops", 1900.0)
    sus = peaks.get("bf16_tflops_sustained", 1700.0)
    f_nom = value / NOMINAL_BF16_TFLOPS
    return {"frac_of_nominal_peak": f_nom, "nominal_peak_tflops": NOMINAL_BF16_TFLOPS,
            "frac_of_burst_peak": value / burst, "frac_of_sustained_peak": value / sus,
            "peak_source": kind, "target_60pct_of_nominal_met": f_nom >= 0.6}


def max_over_ranks(x, device=None):
    """The largest value of `x` over all ranks of the default process group
    (the value itself when there is no group or one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(fwd_flop, steps, world, ms):
    """Whole-job throughput: every rank ran `steps` fwd+bwd steps of `fwd_flop`
    forward flop each (backward = 2.5x), in at most `ms` milliseconds."""
    return 3.5 * fwd_flop * steps * world / (ms / 1e3) / 1e12


def source_hash():
    """Hash of the backward kernel's code (comments and blank lines removed, so
    that a comment edit does not invalidate counters taken on the same code)."""
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(l.rstrip() for l in text.splitlines() if l.strip())
        h.update(code.encode())
    return h.hexdigest()[:16]


def traffic_workload(a):
    """The workload key under which DRAM counters are stored."""
    return "B=1 H=%d S=%d D=%d %s%s%s" % (
        a.heads, a.seqlen, a.head_dim, "causal" if a.causal else "non-causal",
        {"f16": " fp16", "e4m3": " fp8"}.get(a.dtype, ""), " deterministic dQ" if a.deterministic else "")


def ncu_traffic(kernel_key, workload):
    """Per-launch DRAM bytes from a committed ncu summary, or None when the
    counters were taken on another workload or the kernel source has changed
    since they were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    entries = d.get(kernel_key) or []
    if isinstance(entries, dict):
        entries = [entries]
    for e in entries:
        if e.get("source_hash") == source_hash() and e.get("workload") == workload:
            return e.get("bytes_per_launch_full")
    return None


# ---------------------------------------------------------------- reference arm

def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    rows = max(64, oracle_sample_rows(a.seqlen) // 4)
    res = cpu_oracle(a, rows, a.warmup + a.steps)
    times = res["times"][a.warmup:]
    t = sum(times) / len(times)
    value = res["flops"] / t / 1e12
    cb = cpu_baseline_entry(a, dict(res, times=times))
    cb["value"] = value
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(a), "B": 1, "H": a.heads, "S": a.seqlen, "D": a.head_dim,
                   "causal": a.causal, "parallelism": "replicas" if a.gpus > 1 else "single",
                   "sample": "each step: fp64 oracle on query rows 0..%d of one head" % (rows - 1)},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------- fp8 forward

def run_fp8_forward(a):
    """--dtype e4m3: the fp8 forward alone.  One step = the V transpose and the
    forward kernel; metric fwd TFLOP/s against the fp8 peak, taken as twice
    the measured bf16 peak (the nominal dense ratio 4.5 / 2.25 PFLOP/s)."""
    import torch
    from softmax_attention_numerics_gb300 import _lib, attn_fwd_fp8, fwd_fp8_workspace_bytes
    from softmax_attention_numerics_gb300 import build as _build
    if not os.path.exists(_build.LIB):
        _build.build()
    lib = _lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B, H, S, D = 1, a.heads, a.seqlen, 128
    g = torch.Generator(device=dev).manual_seed(42)

    def fp8(x):
        d = float(x.abs().max()) / 448.0
        return (x / d).to(torch.float8_e4m3fn), d

    (q, dq_), (k, dk_), (v, dv_) = (fp8(torch.randn(B, S, H, D, generator=g, device=dev))
                                    for _ in range(3))
    out = torch.empty(B, S, H, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=dev)
    ws = torch.empty(fwd_fp8_workspace_bytes(k), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        attn_fwd_fp8(q, k, v, dq_, dk_, dv_, causal=a.causal, out=out, lse=lse, workspace=ws,
                     stream=stream)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(a.steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in ev:            # torch creates the CUDA event handles on first record
            e0.record(stream)
            e1.record(stream)
        for _ in range(a.warmup):
            step()
    stream.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = lib.attn_launch_count()
    with ClockSampler(0) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(a.steps):
                lib.attn_profile_events(_lib.ATTN_STAGE_FWD, ctypes_ptr(ev[i][0]), ctypes_ptr(ev[i][1]))
                step()
            t1.record(stream)
        lib.attn_profile_events(_lib.ATTN_STAGE_FWD, None, None)
        stream.synchronize()
    launches = lib.attn_launch_count() - launches0
    ms = t0.elapsed_time(t1)
    ff = fwd_flops(B, H, S, D, a.causal)
    value = ff * a.steps / (ms / 1e3) / 1e12
    kern_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    achieved = ff / (kern_ms / 1e3) / 1e12
    peaks, kind = measured_peaks()
    peak = 2.0 * peaks.get("bf16_tflops_sustained", 1700.0)
    nonfinite = sum(int((~torch.isfinite(t.float())).sum()) for t in (out, lse))

    # e2e: host fp8 inputs in, out and lse back, copies inside the timed region
    host_in = [t.view(torch.uint8).cpu().pin_memory() for t in (q, k, v)]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (out, lse)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    e_steps = max(1, min(a.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream), ClockSampler(0) as e_clk:
        e0.record(stream)
        for _ in range(e_steps):
            for dst, src in zip((q, k, v), host_in):
                dst.view(torch.uint8).copy_(src, non_blocking=True)
            step()
            for dst, src in zip(host_out, (out, lse)):
                dst.copy_(src, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e_ms = e0.elapsed_time(e1)
    line = {
        "metric": "attention fwd TFLOP/s, fp8 E4M3 inputs (bf16 out)", "value": value,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms / a.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": "long_seq B=1 H=%d S=%d D=128 %s fwd fp8" % (
                       H, S, "causal" if a.causal else "non-causal"),
                   "B": B, "H": H, "S": S, "D": D, "causal": a.causal, "parallelism": "single",
                   "l2": "no flush: every input tensor (%d MiB) exceeds L2" % (q.numel() >> 20)},
        "roofline": {"bound": "tensor", "kernel": "fwd_fp8", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": "2 x %s bf16_tflops_sustained" % kind},
        "cpu_baseline": None,
        "e2e": {"value": ff * e_steps / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
                "clocks": e_clk.summary()},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "extra": {"fwd_kernel_ms": kern_ms, "nonfinite_outputs": nonfinite},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------- score recompute

def run_score(a):
    """--workload score: attention targets recomputed from the forward's lse
    and summed over the query heads, with the L1 norm of every row.  One step =
    attn_score_recompute (the tile kernel and its L1 reduction) on a resident
    q, k and lse.  Work: 2 D flop per (query, key, head) on the tensor cores
    (halved when causal) and one exp2 per term; the fp32 score is written once."""
    import torch
    from softmax_attention_numerics_gb300 import _lib, attn_fwd, attn_score_recompute
    from softmax_attention_numerics_gb300 import build as _build
    if not os.path.exists(_build.LIB):
        _build.build()
    lib = _lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B, H, S, D = 1, a.heads, a.seqlen, a.head_dim
    Hkv = a.kv_heads if a.kv_heads > 0 else 1
    g = torch.Generator(device=dev).manual_seed(42)
    q = torch.randn(B, S, H, D, generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn(B, S, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
    _, lse = attn_fwd(q, k, k, causal=a.causal)
    score = torch.empty(B, S, S, dtype=torch.float32, device=dev)
    l1 = torch.empty(B, S, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        attn_score_recompute(q, k, lse, causal=a.causal, score=score, l1=l1, stream=stream)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(a.steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            e0.record(stream)
            e1.record(stream)
        for _ in range(a.warmup):
            step()
    stream.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = lib.attn_launch_count()
    with ClockSampler(0) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(a.steps):
                lib.attn_profile_events(_lib.ATTN_STAGE_SCORE, ctypes_ptr(ev[i][0]),
                                        ctypes_ptr(ev[i][1]))
                step()
            t1.record(stream)
        lib.attn_profile_events(_lib.ATTN_STAGE_SCORE, None, None)
        stream.synchronize()
    launches = lib.attn_launch_count() - launches0
    ms = t0.elapsed_time(t1)
    flops = 2.0 * B * S * S * H * D / (2 if a.causal else 1)
    value = flops * a.steps / (ms / 1e3) / 1e12
    kern_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    achieved = flops / (kern_ms / 1e3) / 1e12
    peaks, kind = measured_peaks()
    peak = peaks.get("bf16_tflops", 1900.0)
    out_bytes = 4.0 * B * S * S
    nonfinite = int((~torch.isfinite(score)).sum()) + int((~torch.isfinite(l1)).sum())
    l1_err = float((l1 - H).abs().max())
    # e2e: q, k, lse from pinned host memory in, score and l1 back, every step
    host_in = [t.cpu().pin_memory() for t in (q, k, lse)]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (score, l1)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    e_steps = max(1, min(a.steps, 3))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e_steps):
            for dst, src in zip((q, k, lse), host_in):
                dst.copy_(src, non_blocking=True)
            step()
            for dst, src in zip(host_out, (score, l1)):
                dst.copy_(src, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e_ms = e0.elapsed_time(e1)
    line = {
        "metric": "attention score recompute TFLOP/s (head-summed exp2 targets + L1 norm)",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms / a.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "score_recompute B=%d Hq=%d Hkv=%d S=%d D=%d %s" % (
                       B, H, Hkv, S, D, "causal" if a.causal else "non-causal"),
                   "B": B, "Hq": H, "Hkv": Hkv, "S": S, "D": D, "causal": a.causal,
                   "parallelism": "single",
                   "l2": "no flush: the fp32 score (%d MiB) exceeds L2" % (out_bytes / 2 ** 20)},
        "roofline": {"bound": "tensor", "kernel": "score_sm100", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": "%s bf16_tflops" % kind,
                     "score_write_gbs": out_bytes / (kern_ms / 1e3) / 1e9},
        "cpu_baseline": None,
        "e2e": {"value": flops * e_steps / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "extra": {"kernel_ms": kern_ms, "nonfinite_outputs": nonfinite,
                  "l1_max_abs_err_vs_head_count": l1_err},
    }
    print(json.dumps(line))


def sparse_inputs(B, S, Skv, H, D, K, seed, dev):
    """Seeded sparse-workload inputs drawn on the device (the same recipe as
    attn_workloads.dsa_case: N(0,1) q, kv, dout; K distinct uniform rows per
    token; N(0,1) sink), plus the forward's out and lse from plain torch
    products in fp32 (input preparation, not timed)."""
    import torch
    g = torch.Generator(device=dev).manual_seed(seed)
    q = torch.randn(B, S, H, D, generator=g, device=dev).to(torch.bfloat16)
    kv = torch.randn(B, Skv, D, generator=g, device=dev).to(torch.bfloat16)
    dout = torch.randn(B, S, H, 512, generator=g, device=dev).to(torch.bfloat16)
    idx = torch.rand(B, S, Skv, generator=g, device=dev).argsort(dim=2)[:, :, :K]
    idx = idx.to(torch.int32).contiguous()
    sink = torch.randn(H, generator=g, device=dev)
    scale = 1.0 / math.sqrt(D)
    out = torch.empty(B, S, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, S, H, dtype=torch.float32, device=dev)
    for b in range(B):
        ksel = kv[b].float()[idx[b].long()]                                # [S, K, D]
        s_ = torch.einsum("shd,skd->shk", q[b].float(), ksel) * scale
        logits = torch.cat([s_, sink.view(1, H, 1).expand(S, H, 1)], dim=2)
        lse[b] = torch.logsumexp(logits, dim=2)
        w = torch.exp(s_ - lse[b][..., None])
        out[b] = torch.einsum("shk,skd->shd", w, ksel[..., :512]).to(torch.bfloat16)
    return dict(q=q, kv=kv, out=out, dout=dout, lse=lse, idx=idx, sink=sink, scale=scale)


def sparse_cpu_baseline(D, K, tokens=2048, seed=42):
    """The fp64 oracle on `tokens` tokens of the same shapes (S_kv = 2048,
    H = 64, full index lists, a sink), in this process before any GPU work."""
    import numpy as np
    from oracle import sparse_oracle as OS
    rng = np.random.default_rng(seed)
    S, Skv, H = tokens, 2048, 64
    q = rng.standard_normal((1, S, H, D)).astype(np.float32).astype(np.float64)
    kv = rng.standard_normal((1, Skv, D)).astype(np.float32).astype(np.float64)
    do = rng.standard_normal((1, S, H, 512)).astype(np.float32).astype(np.float64)
    idx = np.stack([rng.permutation(Skv)[:K] for _ in range(S)])[None].astype(np.int32)
    sink = rng.standard_normal(H)
    t0 = time.perf_counter()
    OS.dsa_bwd(q, kv, do, idx, None, sink, scale=1.0 / math.sqrt(D), dv=512)
    dt = time.perf_counter() - t0
    flops = S * K * H * (6.0 * D + 4.0 * 512)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count() or 1,
            "kind": "oracle",
            "sample": "fp64 numpy oracle (forward + backward) of %d tokens x %d entries x %d heads, "
                      "D=%d, S_kv=2048, with a sink (%.3g flop in %.2f s)" % (S, K, H, D, flops, dt)}


def run_sparse(a):
    """--workload sparse: the sparse top-k (DSA) backward with an attention
    sink at the shape of NVIDIA/cudnn-frontend PR #429's check (S = 512
    queries over S_kv = 2048 kv rows, H = 64, D = 576 / values 512, top-k =
    128), `--sparse-batch` sequences per step.  One step = attn_sparse_bwd on
    resident inputs (zero-fill, Delta, main kernel, dkv conversion, d_sink).
    Work: (6 D + 4 * 512) flop per (token, entry, head) on the tensor cores."""
    import torch
    cpu = None if a.no_cpu_baseline else sparse_cpu_baseline(a.sparse_dim, a.topk)
    from softmax_attention_numerics_gb300 import _lib, attn_sparse_bwd, sparse_bwd_workspace_bytes
    from softmax_attention_numerics_gb300 import build as _build
    if not os.path.exists(_build.LIB):
        _build.build()
    lib = _lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B, S, Skv, H, D, K = a.sparse_batch, 512, 2048, 64, a.sparse_dim, a.topk
    x = sparse_inputs(B, S, Skv, H, D, K, 42, dev)
    dq = torch.empty_like(x["q"])
    dkv = torch.empty_like(x["kv"])
    ds = torch.empty(H, dtype=torch.float32, device=dev)
    ws = torch.empty(sparse_bwd_workspace_bytes(x["q"], x["kv"], True), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        attn_sparse_bwd(x["q"], x["kv"], x["out"], x["dout"], x["lse"], x["idx"],
                        attn_sink=x["sink"], scale=x["scale"], dq=dq, dkv=dkv, d_sink=ds,
                        workspace=ws, stream=stream)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(a.steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            e0.record(stream)
            e1.record(stream)
        for _ in range(a.warmup):
            step()
    stream.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = lib.attn_launch_count()
    with ClockSampler(0) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(a.steps):
                lib.attn_profile_events(_lib.ATTN_STAGE_SPARSE, ctypes_ptr(ev[i][0]),
                                        ctypes_ptr(ev[i][1]))
                step()
            t1.record(stream)
        lib.attn_profile_events(_lib.ATTN_STAGE_SPARSE, None, None)
        stream.synchronize()
    launches = lib.attn_launch_count() - launches0
    ms = t0.elapsed_time(t1) / a.steps
    kern_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    tokens = B * S
    flops = tokens * K * H * (6.0 * D + 4.0 * 512)
    # algorithmic bytes of the main kernel: q, dout read and dq written once,
    # the kv rows read once, the fp32 dkv accumulator read and written once,
    # the index lists, lse and Delta
    nbytes = (tokens * H * (2 * D * 2 + 512 * 2) + B * Skv * D * (2 + 8) + tokens * K * 4
              + tokens * H * 8)
    peaks, kind = measured_peaks()
    burst, bw = peaks.get("bf16_tflops", 1900.0), peaks.get("hbm_gbs", 6800.0)
    tf = flops / (kern_ms / 1e3) / 1e12
    gbs = nbytes / (kern_ms / 1e3) / 1e9
    t_flop, t_byte = flops / (burst * 1e12), nbytes / (bw * 1e9)
    if t_byte > t_flop:
        roof = {"bound": "hbm", "achieved": gbs, "peak": bw, "unit": "GB/s", "frac": gbs / bw}
    else:
        roof = {"bound": "tensor", "achieved": tf, "peak": burst, "unit": "TFLOP/s", "frac": tf / burst}
    roof.update({"kernel": "sparse_bwd_sm100", "traffic": None, "peak_source": kind,
                 "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                 "tensor_tflops": tf, "tensor_frac": tf / burst, "hbm_gbs": gbs, "hbm_frac": gbs / bw})
    nonfinite = sum(int((~torch.isfinite(t.float())).sum()) for t in (dq, dkv, ds))
    # e2e: every input from pinned host memory, dq / dkv / d_sink back, each step
    names = ("q", "kv", "out", "dout", "lse", "idx", "sink")
    host_in = [x[n].cpu().pin_memory() for n in names]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dkv, ds)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    e_steps = max(1, min(a.steps, 3))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e_steps):
            for n, src in zip(names, host_in):
                x[n].copy_(src, non_blocking=True)
            step()
            for dst, src in zip(host_out, (dq, dkv, ds)):
                dst.copy_(src, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e_ms = e0.elapsed_time(e1) / e_steps
    line = {
        "metric": "sparse top-k attention backward TFLOP/s (dq, dkv, d_sink)",
        "value": flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "dsa_bwd B=%d S=512 S_kv=2048 H=64 D=%d/512 top-k=%d sink" % (B, D, K),
                   "B": B, "S": S, "S_kv": Skv, "H": H, "D": D, "Dv": 512, "topk": K,
                   "sink": True, "topk_length": False, "parallelism": "single",
                   "l2": "no flush: q, dout and dq (%d MiB) exceed L2" % (
                       tokens * H * (2 * D + 512) * 2 / 2 ** 20)},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": flops / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "extra": {"kernel_ms": kern_ms, "nonfinite_outputs": nonfinite,
                  "tokens_per_s": tokens / (ms / 1e3)},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------- our arm

def main():
    a = parse()
    if a.cpu_oracle_sample:
        run_oracle_sample(a)
        return
    if a.impl == "reference":
        run_reference(a)
        return
    if a.workload == "score":
        if int(os.environ.get("WORLD_SIZE", "1")) > 1:
            raise SystemExit("--workload score: one GPU")
        run_score(a)
        return
    if a.workload == "sparse":
        if int(os.environ.get("WORLD_SIZE", "1")) > 1:
            raise SystemExit("--workload sparse: one GPU")
        run_sparse(a)
        return
    if a.dtype == "e4m3":
        if a.head_dim != 128 or a.deterministic or int(os.environ.get("WORLD_SIZE", "1")) > 1:
            raise SystemExit("--dtype e4m3: one GPU, D = 128, forward only")
        run_fp8_forward(a)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # Bind this rank's GPU before the process group so NCCL's communicator and
    # every collective use it.
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    # CPU baseline first: the oracle child process runs before this process
    # touches the GPU heavily (rank 0 at N=1 only).
    cpu_res = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu_res = cpu_oracle(a, oracle_sample_rows(a.seqlen), 2)

    from softmax_attention_numerics_gb300 import _lib, attn_bwd, attn_fwd
    from softmax_attention_numerics_gb300 import build as _build
    if not os.path.exists(_build.LIB):
        _build.build()
    lib = _lib.load()

    B, H, S, D = 1, a.heads, a.seqlen, a.head_dim
    scale = 1.0 / math.sqrt(D)
    g = torch.Generator(device=dev).manual_seed(42 + rank)
    shape = (B, S, H, D)
    q, k, v, do = (torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
                   .to(torch.float16 if a.dtype == "f16" else torch.bfloat16) for _ in range(4))
    stream = torch.cuda.Stream(device=dev)
    ws = torch.empty(max(1, _bwd_ws(q, k)), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step(s):
        attn_fwd(q, k, v, causal=a.causal, scale=scale, out=out, lse=lse, stream=s)
        attn_bwd(q, k, v, out, do, lse, causal=a.causal, scale=scale, dq=dq, dk=dk, dv=dv,
                 workspace=ws, stream=s, deterministic=a.deterministic)

    stages = (_lib.ATTN_STAGE_FWD, _lib.ATTN_STAGE_BWD_PREPROCESS, _lib.ATTN_STAGE_BWD_MAIN,
              _lib.ATTN_STAGE_BWD_DQ)
    ev = {st: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(a.steps)] for st in stages}
    with torch.cuda.stream(stream):
        for st in stages:
            for e0, e1 in ev[st]:
                e0.record(stream)
                e1.record(stream)
        for _ in range(a.warmup):
            step(stream)
    stream.synchronize()

    # Device-timed region.
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = lib.attn_launch_count()
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(a.steps):
                for st in stages:
                    lib.attn_profile_events(st, ctypes_ptr(ev[st][i][0]), ctypes_ptr(ev[st][i][1]))
                step(stream)
            t1.record(stream)
        for st in stages:
            lib.attn_profile_events(st, None, None)
        stream.synchronize()
    launches = lib.attn_launch_count() - launches0
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(t0.elapsed_time(t1), dev)
    if world > 1:
        dist.barrier()

    # Non-finite check of the last step's results.
    nonfinite = sum(int((~torch.isfinite(t.float())).sum()) for t in (out, lse, dq, dk, dv))

    stage_ms = {st: statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev[st]) for st in stages}
    ff = fwd_flops(B, H, S, D, a.causal)
    value = job_tflops(ff, a.steps, world, ms)

    peaks, peak_kind = measured_peaks()
    tensor_peak = peaks.get("bf16_tflops_sustained", 1700.0)
    # main kernel: S, dP, dV, dK (+ dQ unless the per-query-tile kernel does it)
    main_flops = (2.0 if a.deterministic else 2.5) * ff
    main_achieved = main_flops / (stage_ms[_lib.ATTN_STAGE_BWD_MAIN] / 1e3) / 1e12
    traffic = ncu_traffic("bwd_main", traffic_workload(a))
    roofline = {"bound": "tensor", "kernel": "bwd_main", "achieved": main_achieved,
                "peak": tensor_peak, "unit": "TFLOP/s", "frac": main_achieved / tensor_peak,
                "traffic": traffic,
                "peak_source": "%s bf16_tflops_sustained" % peak_kind}
    fwd_tflops = ff / (stage_ms[_lib.ATTN_STAGE_FWD] / 1e3) / 1e12
    pre_bytes = B * H * S * (4 * D + 12)
    dq_bytes = B * H * S * D * 6
    extra = {
        "fwd_kernel_tflops": fwd_tflops,
        "fwd_kernel_frac_of_peak": fwd_tflops / tensor_peak,
        "bwd_main_ms": stage_ms[_lib.ATTN_STAGE_BWD_MAIN],
        "fwd_ms": stage_ms[_lib.ATTN_STAGE_FWD],
        "bwd_preprocess_gbs": pre_bytes / (stage_ms[_lib.ATTN_STAGE_BWD_PREPROCESS] / 1e3) / 1e9,
        "bwd_dq_ms": stage_ms[_lib.ATTN_STAGE_BWD_DQ],
        "dq_convert_gbs": (None if a.deterministic else
                           dq_bytes / (stage_ms[_lib.ATTN_STAGE_BWD_DQ] / 1e3) / 1e9),
        "hbm_peak_gbs": peaks.get("hbm_gbs"),
        "nonfinite_outputs": nonfinite,
    }

    # End-to-end through the public API with host buffers (pinned), copies timed.
    # Pipelined like an input pipeline would be: step i+1's inputs are copied in
    # on one copy stream and step i's outputs copied out on another while the
    # compute stream runs step i+1; inputs and outputs are double-buffered on
    # the device.  The timed region runs from the first input copy to the end of
    # the last output copy, so every step's copies are inside it.
    host_in = [t.cpu().pin_memory() for t in (q, k, v, do)]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (out, lse, dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    dev_in = [[torch.empty_like(t) for t in (q, k, v, do)] for _ in range(2)]
    dev_out = [[out, lse, dq, dk, dv], [torch.empty_like(t) for t in (out, lse, dq, dk, dv)]]
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    new_ev = lambda: torch.cuda.Event()
    done_in = [new_ev() for _ in range(2)]      # inputs of buffer b are on the device
    done_step = [new_ev() for _ in range(2)]    # compute on buffer b finished
    done_out = [new_ev() for _ in range(2)]     # outputs of buffer b are on the host

    def copy_in(i):
        bb = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(done_step[bb])        # step i-2 no longer reads them
            for hdst, hsrc in zip(dev_in[bb], host_in):
                hdst.copy_(hsrc, non_blocking=True)
            done_in[bb].record(s_in)

    def compute(i):
        bb = i % 2
        with torch.cuda.stream(stream):
            stream.wait_event(done_in[bb])
            if i >= 2:
                stream.wait_event(done_out[bb])       # step i-2's outputs left
            qq, kk, vv, dd = dev_in[bb]
            o_, l_, dq_, dk_, dv_ = dev_out[bb]
            attn_fwd(qq, kk, vv, causal=a.causal, scale=scale, out=o_, lse=l_, stream=stream)
            attn_bwd(qq, kk, vv, o_, dd, l_, causal=a.causal, scale=scale, dq=dq_, dk=dk_, dv=dv_,
                     workspace=ws, stream=stream, deterministic=a.deterministic)
            done_step[bb].record(stream)

    def copy_out(i):
        bb = i % 2
        with torch.cuda.stream(s_out):
            s_out.wait_event(done_step[bb])
            for hdst, dsrc in zip(host_out, dev_out[bb]):
                hdst.copy_(dsrc, non_blocking=True)
            done_out[bb].record(s_out)

    def run_pipeline(n, marks=None):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            copy_out(i)
            if marks is not None:
                s_out.wait_stream(stream)
                marks[i + 1].record(s_out)

    e_steps = max(1, min(a.steps, 5))
    run_pipeline(2)                                   # warm-up (host pages, copy engines)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps + 1)]
    with ClockSampler(local) as e_clk:
        marks[0].record(s_in)
        run_pipeline(e_steps, marks)
        torch.cuda.synchronize(dev)
    e_step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(e_steps)]
    e_ms = max_over_ranks(marks[0].elapsed_time(marks[-1]), dev)
    e2e_value = job_tflops(ff, e_steps, world, e_ms)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms / a.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": a.dtype,
            "data": "synthetic",
            "config": {"workload": workload_name(a), "B": B, "H": H, "S": S, "D": D,
                       "causal": a.causal, "parallelism": "replicas" if world > 1 else "single",
                       "l2": "no flush: every input tensor (%d MiB) exceeds L2"
                             % (q.numel() * 2 >> 20),
                       "frac_of_peak": value / tensor_peak,
                       "peaks": peak_fractions(value, peaks, peak_kind)},
            "roofline": roofline,
            "cpu_baseline": cpu_baseline_entry(a, cpu_res) if cpu_res else None,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e_steps,
                    "step_ms": [round(x, 2) for x in e_step_ms], "clocks": e_clk.summary()},
            "gpu_launches": int(launches),
            "clocks": clk.summary(),
            "extra": extra,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def _bwd_ws(q, k):
    from softmax_attention_numerics_gb300 import bwd_workspace_bytes
    return bwd_workspace_bytes(q, k)


def ctypes_ptr(ev):
    import ctypes
    return ctypes.c_void_p(ev.cuda_event)


if __name__ == "__main__":
    main()
