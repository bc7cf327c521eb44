#!/usr/bin/env python3
"""Benchmark of the selective-scan library on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic input.
The headline workload is the flat affine scan over n = 2**28 fp32 elements
(a ~ U(0.9, 1), b ~ N(0, 1), seed 0): inputs are staged in HBM once, then K
timed calls of ss_affine_scan follow W untimed ones. Inputs (3.2 GB with the
output) are larger than L2, so no flush is needed between calls. The three
S6 workloads are timed the same way (with an L2 flush between calls where
their bytes fit in L2) and reported under "per_config".

Rank 0 prints one JSON line. With --gpus N > 1 (under torchrun) every rank
runs its own replica: the path has no exchange step, so there is no
collective on the data path; value is the work of all ranks over the
slowest rank's time.

--impl reference times the float64 CPU oracle (the only reference this
problem has) on a bounded sample of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "selective-scan elements/s, HBM GB/s and % of GB300 roofline (1 GPU)"
HEADLINE = "affine_large"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "linear_recurrences_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str, src_hash: str):
    """dram bytes per launch from the committed ncu summary, or None when the
    kernel changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    e = data.get(f"{kernel}/{workload}")
    if not e or e.get("source_hash") != src_hash:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows
                                                         if r[3].replace(".", "").isdigit())}


def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` over the ranks of the default process group (the job's
    time is its slowest rank's); returns `value` when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- device timing
def time_launches(torch, fn, steps, warmup, stream, flush=None, barrier=None):
    """Per-launch CUDA-event durations (ms) of `fn` over `steps` timed calls,
    plus the wall-to-wall event time of the whole timed region."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            if flush is not None:
                flush()
            fn()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        region0.record(stream)
        for i in range(steps):
            if flush is not None:
                flush()
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
        region1.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return per, region0.elapsed_time(region1)


def hbm_copy_probe(torch, dev):
    """Sentinel: copy of 1 GiB (bf16), read + write bytes over the best time."""
    a = torch.empty(1 << 29, dtype=torch.bfloat16, device=dev).fill_(1.0)
    b = torch.empty_like(a)
    best = None
    for _ in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        best = t if best is None else min(best, t)
    del a, b
    return 2 * (1 << 30) / (best * 1e-3) / 1e9


def mufu_probe(torch, ss, dev, sms):
    """ex2 operations per second on the special-function unit."""
    blocks, iters = sms * 8, 4096
    out = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    ss.ss_probe_mufu_ex2(out, blocks, iters)
    torch.cuda.synchronize()
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        ss.ss_probe_mufu_ex2(out, blocks, iters)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        best = t if best is None else min(best, t)
    ops = blocks * 256 * 8 * iters
    return ops / (best * 1e-3)


# ---------------------------------------------------------------- workloads
def affine_setup(torch, dev, name):
    import workloads
    w = workloads.AFFINE[name]
    a, b = workloads.affine_inputs(w.n, w.a_lo, w.a_hi)
    return w, a, b, torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)


def s6_bytes_and_ops(w):
    es = 2 if w.io == "bf16" else 4
    B, L, D, N = w.B, w.L, w.D, w.N
    byts = 3 * es * B * L * D + 2 * es * B * L * N + 4 * D * N + 4 * D
    mufu = B * L * D * N + (2 * B * L * D if w.softplus else 0)
    return byts, mufu


def s6_variant(name):
    """(workload, variant) for an S6 bench name: "s6_x", "s6_x_state" or
    "s6_x_bwd"."""
    import workloads
    for suffix in ("_state", "_bwd", "_layer"):
        if name.endswith(suffix) and name[: -len(suffix)] in workloads.S6:
            return workloads.S6[name[: -len(suffix)]], suffix[1:]
    return workloads.S6[name], ""


def bench_s6(torch, ss, dev, name, steps, warmup, stream, hbm_peak, sfu_peak, cpu=False):
    """One S6 workload. A name ending in "_state" runs the forward-with-state
    call from a seeded random h0, writing h_last (2 x B*D*N*4 more bytes); one
    ending in "_bwd" runs the backward pass for a seeded random dy: reads x,
    delta, dy, Bt, Ct once and writes dx, ddelta (storage type) and dBt, dCt,
    dA, dDskip (fp32); MUFU ops BLDN + (3 BLD with softplus: softplus and its
    sigmoid)."""
    import numpy as np
    import workloads
    w, variant = s6_variant(name)
    state = variant == "state"
    inp = workloads.s6_workload_inputs(w)

    def t(v):
        x = torch.from_numpy(v)
        if inp.io == "bf16" and v.dtype.name == "uint16":
            x = x.view(torch.bfloat16)
        return x.to(dev)

    args = (t(inp.x), t(inp.delta), t(inp.Bt), t(inp.Ct), t(inp.A), t(inp.Dskip))
    y = torch.empty_like(args[0])
    fn = ss.ss_selective_scan_bidir if w.bidir else ss.ss_selective_scan_fwd
    call = lambda: fn(*args, delta_softplus=w.softplus, y=y, stream=stream)
    byts, mufu = s6_bytes_and_ops(w)
    if state:
        g = np.random.Generator(np.random.PCG64(7))
        h0 = torch.from_numpy(g.standard_normal((w.B, w.D, w.N)).astype(np.float32)).to(dev)
        h_last = torch.empty_like(h0)
        call = lambda: ss.ss_selective_scan_fwd_state(*args, h0=h0, delta_softplus=w.softplus,
                                                      y=y, h_last=h_last, stream=stream)
        byts += 2 * 4 * w.B * w.D * w.N
    t_gemm = 0.0
    if variant == "layer":
        # projections of the workload's shape with seeded random weights:
        # W ~ N(0, 1/D), b_delta ~ N(-4, 1) (steps like the workload's)
        g = np.random.Generator(np.random.PCG64(23))
        W_np = (g.standard_normal((w.D + 2 * w.N, w.D)) / np.sqrt(w.D)).astype(np.float32)
        W = t(W_np)
        if inp.io == "bf16":
            W = W.to(torch.bfloat16)
            W_np = W.float().cpu().numpy()  # the values the GPU sees
        bd_np = g.normal(-4.0, 1.0, w.D).astype(np.float32)
        bd = torch.from_numpy(bd_np).to(dev)
        io_dtype = ss.SS_BF16 if w.io == "bf16" else ss.SS_F32
        lws = ss.new_workspace(
            ss.ss_selective_scan_layer_workspace_bytes(w.B, w.L, w.D, w.N, io_dtype), dev)
        call = lambda: ss.ss_selective_scan_layer_fwd(args[0], W, bd, args[4], args[5], y=y,
                                                      workspace=lws, stream=stream)
        es = 2 if w.io == "bf16" else 4
        M = w.B * w.L
        gemm_flops = 2.0 * M * w.D * (w.D + 2 * w.N)
        peaks, _ = measured_peaks()
        t_gemm = gemm_flops / (float(peaks.get("bf16_tflops", 1900.0)) * 1e12)
        # x and W read, projections written and read back by the scan
        byts += es * (w.D + 2 * w.N) * w.D + 2 * es * M * (w.D + 2 * w.N)
    if variant == "bwd":
        g = np.random.Generator(np.random.PCG64(17))
        dy = t(g.standard_normal((w.B, w.L, w.D)).astype(np.float32))
        if inp.io == "bf16":
            dy = dy.to(torch.bfloat16)
        ws = ss.new_workspace(ss.ss_selective_scan_bwd_workspace_bytes(w.B, w.L, w.D, w.N), dev)
        call = lambda: ss.ss_selective_scan_bwd(*args, dy, delta_softplus=w.softplus,
                                                workspace=ws, stream=stream)
        es = 2 if w.io == "bf16" else 4
        BLD, BLN = w.B * w.L * w.D, w.B * w.L * w.N
        byts = 5 * es * BLD + 2 * es * BLN + 2 * 4 * BLN + 4 * (2 * w.D * w.N + 2 * w.D)
        mufu = BLD * w.N + (3 * BLD if w.softplus else 0)
    flush = None
    if byts < 2 * L2_BYTES:
        junk = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        flush = lambda: junk.fill_(0.0)
    per, _ = time_launches(torch, call, steps, warmup, stream, flush=flush)
    ms = statistics.mean(per)
    base = None
    if cpu:
        base = s6_oracle_baseline(w, variant, inp, (W_np, bd_np) if variant == "layer" else None)
    t_hbm = byts / (hbm_peak * 1e9)
    t_sfu = mufu / sfu_peak
    t_roof = max(t_hbm, t_sfu) + t_gemm
    return {
        "elements": w.elements, "shape": [w.B, w.L, w.D, w.N], "io": w.io,
        "softplus": w.softplus, "bidir": w.bidir, "variant": variant or "forward", "ms": ms,
        "ms_min": min(per),
        "elements_per_s": w.elements / (ms * 1e-3),
        "gbs": byts / (ms * 1e-3) / 1e9, "algorithmic_bytes": byts, "mufu_ops": mufu,
        "t_hbm_us": t_hbm * 1e6, "t_sfu_us": t_sfu * 1e6,
        **({"t_gemm_us": t_gemm * 1e6, "gemm_peak": "measured bf16_tflops"} if t_gemm else {}),
        "bound": "hbm" if t_hbm >= t_sfu else "sfu",
        "roofline_frac": t_roof / (ms * 1e-3),
        "l2": "flushed between calls" if flush else "inputs larger than L2",
        "workspace_bytes": (
            ss.ss_selective_scan_bwd_workspace_bytes(w.B, w.L, w.D, w.N) if variant == "bwd" else
            ss.ss_selective_scan_layer_workspace_bytes(
                w.B, w.L, w.D, w.N, ss.SS_BF16 if w.io == "bf16" else ss.SS_F32)
            if variant == "layer" else
            ss.ss_selective_scan_workspace_bytes(w.B, w.L, w.D, w.N,
                                                 ss.SS_BF16 if w.io == "bf16" else ss.SS_F32,
                                                 w.bidir)),
        **({"cpu_baseline": base} if base else {}),
    }


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def s6_oracle_baseline(w, variant, inp, layer=None, elems_target=3_000_000):
    """The float64 oracle, as it stands, on a bounded sample of one S6
    workload: batch element 0 and its first Ls steps, Ls chosen so that the
    sample holds about `elems_target` (b, t, d) elements (fewer for the
    bidirectional and backward passes, which do more per element). Timed on
    one thread and on every core this process may run on. Returns the
    cpu_baseline object for that config's per_config entry."""
    import numpy as np
    import oracle
    lib = oracle.load()
    per_elem = {"bwd": 3, "layer": 1}.get(variant, 2 if w.bidir else 1)
    Ls = max(1, min(w.L, elems_target // per_elem // w.D))
    sl = lambda v: np.ascontiguousarray(v[:1, :Ls])
    x, dl, Bt, Ct = sl(inp.x_f32), sl(inp.delta_f32), sl(inp.Bt_f32), sl(inp.Ct_f32)
    g = np.random.Generator(np.random.PCG64(7))
    dy = g.standard_normal((1, Ls, w.D)).astype(np.float32)
    h0 = g.standard_normal((1, w.D, w.N))

    def call(threads):
        if variant == "bwd":
            return oracle.s6_bwd(x, dl, Bt, Ct, inp.A, inp.Dskip, dy, softplus=w.softplus,
                                 threads=threads, lib=lib)
        if variant == "state":
            return oracle.s6_fwd_state(x, dl, Bt, Ct, inp.A, inp.Dskip, h0=h0,
                                       softplus=w.softplus, threads=threads, lib=lib)
        if variant == "layer":
            W, b = layer
            return oracle.layer_fwd(x, W, b, inp.A, inp.Dskip, io=w.io, threads=threads, lib=lib)
        f = oracle.s6_bidir if w.bidir else oracle.s6_fwd
        return f(x, dl, Bt, Ct, inp.A, inp.Dskip, softplus=w.softplus, threads=threads, lib=lib)

    cores = host_cores()
    rates = {}
    for threads in (1, cores):
        t0 = time.perf_counter()
        call(threads)
        rates[threads] = Ls * w.D / (time.perf_counter() - t0)
    what = {"bwd": "backward (every gradient)", "state": "forward from a state, h_last",
            "layer": "projections (float64 numpy matmul) + scan"}.get(
        variant, "bidirectional" if w.bidir else "forward")
    return {"value": rates[cores], "unit": "elements/s", "cores": cores, "kind": "oracle",
            "value_1_thread": rates[1], "host_cores": cores,
            "sample": f"batch element 0, first {Ls} of {w.L} steps ({Ls * w.D} elements) of "
                      f"the workload's inputs; {what}, float64, timed once on 1 thread and "
                      f"once on {cores} threads (channels split across threads)"}


def bench_proj_gemm(torch, ss, dev, steps, warmup, stream):
    """The bf16 layer's projection GEMM alone (tcgen05 kernel, bias in the
    epilogue) at the bf16 workload's layer shape: M = B*L = 32768, K = D =
    1536, Nout = D + 2N = 1568; 2 M K Nout flops per call."""
    import numpy as np
    import workloads
    w = workloads.S6["s6_bf16"]
    M, K, Nout = w.B * w.L, w.D, w.D + 2 * w.N
    g = np.random.Generator(np.random.PCG64(29))
    x = torch.from_numpy(g.standard_normal((M, K)).astype(np.float32)).to(dev).to(torch.bfloat16)
    W = torch.from_numpy((g.standard_normal((Nout, K)) / np.sqrt(K)).astype(np.float32)).to(
        dev).to(torch.bfloat16)
    bias = torch.from_numpy(g.normal(-4.0, 1.0, K).astype(np.float32)).to(dev)
    out = torch.empty((M, Nout), dtype=torch.bfloat16, device=dev)
    ws = ss.new_workspace(256, dev)
    per, _ = time_launches(torch, lambda: ss.ss_testing_proj_gemm(x, W, bias=bias, out=out,
                                                                  workspace=ws, stream=stream),
                           steps, warmup, stream)
    if ss.ss_get_device_status(ws) != ss.SS_OK:
        raise RuntimeError("device reported an error in the projection GEMM")
    ms = statistics.mean(per)
    flops = 2.0 * M * K * Nout
    peaks, kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    tf = flops / (ms * 1e-3) / 1e12
    # for context, not a product path: the vendor library's plain bf16 GEMM
    # (torch.mm, no bias) on the same operands and shape, timed the same way
    # (after this kernel's own timing; a failure here is recorded, not raised)
    library = {"what": "torch.mm bf16 (cuBLAS), no bias"}
    try:
        WT = W.t()
        lib_per, _ = time_launches(torch, lambda: torch.mm(x, WT, out=out), steps, warmup, stream)
        lib_ms = statistics.mean(lib_per)
        library.update(ms=lib_ms, tflops=flops / (lib_ms * 1e-3) / 1e12)
    except Exception as e:  # noqa: BLE001 - context figure only
        library["error"] = f"{type(e).__name__}: {e}"[:200]
    return {"shape": [M, K, Nout], "ms": ms, "ms_min": min(per), "tflops": tf,
            "bound": "tensor", "peak_tflops": peak, "peak_source": f"{kind} bf16_tflops",
            "roofline_frac": tf / peak, "kernel": "proj_gemm_kernel (tcgen05, TMA, bias epilogue)",
            "library_same_shape": library,
            "l2": "inputs (100 MB x + 4.8 MB W) near L2 size, no flush"}


def round_floats(v, digits=5):
    """The JSON line with floats at `digits` significant digits (the timing
    noise is larger), so the line stays short enough to read whole."""
    if isinstance(v, float):
        return float(f"{v:.{digits}g}")
    if isinstance(v, dict):
        return {k: round_floats(x, digits) for k, x in v.items()}
    if isinstance(v, list):
        return [round_floats(x, digits) for x in v]
    return v


def config_summary(per_cfg, line):
    """One short entry per workload, the five configurations of the problem
    last: time per call, fraction of its roofline, and the oracle's rate on
    one thread and on every core (elements/s) beside the GPU's."""
    order = ["proj_gemm_bf16", "affine_large_log_step", "s6_bf16_state", "s6_fp32_bwd",
             "s6_bf16_bwd", "s6_bf16_layer", "affine_small_graph",
             "affine_small", "affine_large", "s6_fp32", "s6_bf16", "s6_bidir"]
    out = {}
    for name in order:
        e = per_cfg.get(name)
        if not e:
            continue
        r = {"ms": e.get("ms")}
        if e.get("roofline_frac") is not None:
            r["roofline_frac"] = e["roofline_frac"]
        if e.get("elements_per_s") is not None:
            r["elem_per_s"] = e["elements_per_s"]
        cb = e.get("cpu_baseline") or (line.get("cpu_baseline") if name == "affine_large" else None)
        if cb:
            r["oracle_elem_per_s"] = {"1_thread": cb.get("value_1_thread", cb["value"] if cb.get("cores") == 1 else None),
                                      "all_cores": cb["value"] if cb.get("cores", 1) > 1 else None,
                                      "cores": cb.get("host_cores", cb.get("cores"))}
        out[name] = r
    return out


# ---------------------------------------------------------------- arms
def run_reference(args, rank):
    if rank != 0:
        return
    import numpy as np
    import oracle
    import workloads
    w = workloads.AFFINE[HEADLINE]
    sample = 1 << 27
    a, b = workloads.affine_inputs(sample, w.a_lo, w.a_hi)
    lib = oracle.load()
    for _ in range(max(args.warmup, 0)):
        oracle.affine(a[: 1 << 20], b[: 1 << 20], lib=lib)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        h = oracle.affine(a, b, lib=lib)
    dt = time.perf_counter() - t0
    assert np.isfinite(h[-1])
    value = sample * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "elements/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE, "n_per_step": sample, "n_workload": w.n,
                   "a": "U(0.9,1)", "b": "N(0,1)", "seed": 0},
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": 1, "kind": "oracle",
                         "sample": f"first 2**27 of the {HEADLINE} inputs per step, "
                                   "sequential float64 loop, one thread"},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(budget_s: float):
    """The oracle as it stands, on the headline input, on this host."""
    import oracle
    import workloads
    w = workloads.AFFINE[HEADLINE]
    a, b = workloads.affine_inputs(w.n, w.a_lo, w.a_hi)
    lib = oracle.load()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.affine(a, b, lib=lib)
        reps += 1
        if time.perf_counter() - t0 >= budget_s or reps >= 20:
            break
    dt = time.perf_counter() - t0
    return {"value": w.n * reps / dt, "unit": "elements/s", "cores": 1, "kind": "oracle",
            "host_cores": host_cores(),
            "sample": f"full {HEADLINE} input (2**28 elements) x {reps} passes, sequential "
                      "float64 loop, one thread (the recurrence is sequential)"}


def run_ours(args, rank, world, local_rank):
    import torch
    import linear_recurrences_gb300 as ss
    from linear_recurrences_gb300 import build as ssbuild
    ssbuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        barrier = dist.barrier
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))

    w, a_np, b_np, a, b = affine_setup(torch, dev, HEADLINE)
    h = torch.empty_like(a)
    ws = ss.new_workspace(ss.ss_affine_scan_workspace_bytes(w.n), dev)
    call = lambda: ss.ss_affine_scan(a, b, h, workspace=ws, stream=stream)

    with ClockSampler(local_rank) as clk:
        per, region_ms = time_launches(torch, call, args.steps, args.warmup, stream,
                                       barrier=barrier)
    status = ss.ss_get_device_status(ws, stream)
    if status != ss.SS_OK:
        raise RuntimeError(f"device reported {ss.ss_status_string(status)}")
    clocks = clk.summary()
    region_ms_all = max_over_ranks(region_ms, dev)
    elems = w.n * args.steps * world
    value = elems / (region_ms_all * 1e-3)
    launch_ms = statistics.mean(per)
    alg_bytes = 12 * w.n
    achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
    src = source_hash("affine_scan.cu", "ss_common.cuh")

    # end to end through the C ABI with host buffers: H2D inputs, scan, D2H output
    a_host = torch.from_numpy(a_np).pin_memory()
    b_host = torch.from_numpy(b_np).pin_memory()
    h_host = torch.empty(w.n, dtype=torch.float32).pin_memory()

    hws = ss.new_workspace(ss.ss_affine_scan_host_workspace_bytes(w.n), dev)

    def e2e_step():  # the library's host-buffer entry: chunked, copies overlapped
        ss.ss_affine_scan_host(a_host, b_host, h_host, workspace=hws, stream=stream)

    def serial_step():  # for comparison: whole-array copies around one scan
        a.copy_(a_host, non_blocking=True)
        b.copy_(b_host, non_blocking=True)
        ss.ss_affine_scan(a, b, h, workspace=ws, stream=stream)
        h_host.copy_(h, non_blocking=True)

    e2e_steps = max(3, args.steps // 4)
    e2e_per, e2e_region = time_launches(torch, e2e_step, e2e_steps, min(args.warmup, 3), stream,
                                        barrier=barrier)
    e2e_value = w.n * len(e2e_per) * world / (max_over_ranks(e2e_region, dev) * 1e-3)
    if ss.ss_get_device_status(hws, stream) != ss.SS_OK:
        raise RuntimeError("device reported an error in the host-buffer scan")
    ser_per, ser_region = time_launches(torch, serial_step, e2e_steps, min(args.warmup, 3), stream,
                                        barrier=barrier)
    serial_value = w.n * len(ser_per) * world / (max_over_ranks(ser_region, dev) * 1e-3)
    del hws

    extras = {}
    if rank == 0 and not args.no_extras:
        sfu = mufu_probe(torch, ss, dev, sms)
        extras["sfu_probe_ex2_per_s"] = sfu
        if clocks.get("sm_mhz"):
            extras["sfu_probe_ex2_per_clk_per_sm"] = sfu / (clocks["sm_mhz"] * 1e6) / sms
        extras["hbm_probe_gbs"] = hbm_copy_probe(torch, dev)
        per_cfg = {}
        small_w, *_rest, sa, sb = affine_setup(torch, dev, "affine_small")
        sh = torch.empty_like(sa)
        sws = ss.new_workspace(ss.ss_affine_scan_workspace_bytes(small_w.n), dev)
        junk = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        sper, _ = time_launches(torch, lambda: ss.ss_affine_scan(sa, sb, sh, workspace=sws,
                                                                 stream=stream),
                                args.steps, args.warmup, stream, flush=lambda: junk.fill_(0.0))
        del junk
        sms_ = statistics.mean(sper)
        per_cfg["affine_small"] = {"elements": small_w.n, "ms": sms_,
                                   "elements_per_s": small_w.n / (sms_ * 1e-3),
                                   "gbs": 12 * small_w.n / (sms_ * 1e-3) / 1e9,
                                   "bound": "launch latency", "l2": "flushed between calls"}
        if not args.no_cpu:
            import oracle
            a_s, b_s = _rest[0], _rest[1]
            olib, reps, t0 = oracle.load(), 0, time.perf_counter()
            while time.perf_counter() - t0 < 0.5:
                oracle.affine(a_s, b_s, lib=olib)
                reps += 1
            per_cfg["affine_small"]["cpu_baseline"] = {
                "value": small_w.n * reps / (time.perf_counter() - t0), "unit": "elements/s",
                "cores": 1, "kind": "oracle", "host_cores": host_cores(),
                "sample": f"the full affine_small input x {reps} passes, sequential float64 "
                          "loop, one thread"}
        # the same small scan replayed from a CUDA graph of 10 launches
        # (launch overhead amortised; inputs stay in L2 between launches)
        gs = torch.cuda.Stream(dev)
        with torch.cuda.stream(gs):
            ss.ss_affine_scan(sa, sb, sh, workspace=sws, stream=gs)
        gs.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(10):
                ss.ss_affine_scan(sa, sb, sh, workspace=sws, stream=gs)
        gper, _ = time_launches(torch, graph.replay, args.steps, args.warmup, gs)
        gms = statistics.mean(gper) / 10
        per_cfg["affine_small_graph"] = {"elements": small_w.n, "ms": gms,
                                         "elements_per_s": small_w.n / (gms * 1e-3),
                                         "gbs": 12 * small_w.n / (gms * 1e-3) / 1e9,
                                         "bound": "launch latency",
                                         "l2": "inputs L2-resident (no flush inside the graph)",
                                         "how": "10 launches captured in one CUDA graph, replayed"}
        del graph
        per_cfg[HEADLINE] = {"elements": w.n, "ms": launch_ms,
                             "elements_per_s": w.n / (launch_ms * 1e-3), "gbs": achieved,
                             "bound": "hbm", "roofline_frac": achieved / hbm_peak}
        # comparison kernel: the same scan with log-step (Hillis-Steele) tiles
        lws = ss.new_workspace(ss.ss_affine_scan_workspace_bytes(w.n), dev)
        lper, _ = time_launches(
            torch, lambda: ss.ss_affine_scan_log_step(a, b, h, workspace=lws, stream=stream),
            args.steps, args.warmup, stream)
        lms = statistics.mean(lper)
        per_cfg[HEADLINE + "_log_step"] = {
            "elements": w.n, "ms": lms, "elements_per_s": w.n / (lms * 1e-3),
            "gbs": 12 * w.n / (lms * 1e-3) / 1e9, "roofline_frac": 12 * w.n / (lms * 1e-3) / 1e9 / hbm_peak,
            "kernel": "comparison: log-step (Hillis-Steele) tile scan, same look-back"}
        del lws
        per_cfg["proj_gemm_bf16"] = bench_proj_gemm(torch, ss, dev, args.steps, args.warmup,
                                                    stream)
        for name in ("s6_fp32", "s6_bf16", "s6_bidir", "s6_bf16_state", "s6_fp32_bwd",
                     "s6_bf16_bwd", "s6_bf16_layer"):
            per_cfg[name] = bench_s6(torch, ss, dev, name, args.steps, args.warmup, stream,
                                     hbm_peak, sfu, cpu=not args.no_cpu)
        extras["per_config"] = per_cfg

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": region_ms_all / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": HEADLINE, "n": w.n, "a": "U(0.9,1)", "b": "N(0,1)", "seed": 0,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (3.2 GB per call), no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": committed_traffic("affine_scan_kernel", HEADLINE, src),
                     "kernel": "affine_scan_kernel", "algorithmic_bytes_per_launch": alg_bytes,
                     "avg_launch_ms": launch_ms},
        "cpu_baseline": cpu_baseline(args.cpu_seconds) if world == 1 else None,
        "e2e": {"value": e2e_value, "unit": "elements/s", "h2d_bytes_per_step": 8 * w.n,
                "d2h_bytes_per_step": 4 * w.n, "api": "ss_affine_scan_host (pinned host a, b, h)",
                "ms_per_step": statistics.mean(e2e_per),
                "serial_copies": {"value": serial_value, "ms_per_step": statistics.mean(ser_per),
                                  "how": "whole-array copies, one ss_affine_scan, copy back"}},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "source_hash": src,
    }
    line.update(extras)
    if "per_config" in extras:
        line["summary"] = config_summary(extras["per_config"], line)
    print(json.dumps(round_floats(line)), flush=True)


def run_single(args):
    """One workload's timed loop on this GPU (used for per-kernel timing and
    for ncu captures); prints one JSON line for that workload."""
    import torch
    import workloads
    import linear_recurrences_gb300 as ss
    from linear_recurrences_gb300 import build as ssbuild
    ssbuild.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    peaks, _ = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    name = args.workload
    if name in workloads.S6 or any(name.endswith(x) and name[: -len(x)] in workloads.S6
                                   for x in ("_state", "_bwd", "_layer")):
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        sfu = mufu_probe(torch, ss, dev, sms) if not args.no_extras else 9.86e12
        r = bench_s6(torch, ss, dev, name, args.steps, args.warmup, stream, hbm_peak, sfu)
    elif name == "proj_gemm_bf16":
        r = bench_proj_gemm(torch, ss, dev, args.steps, args.warmup, stream)
    elif name in workloads.AFFINE or (name.endswith("_log_step") and name[:-9] in workloads.AFFINE):
        log_step = name.endswith("_log_step")
        name = name[:-9] if log_step else name
        fn = ss.ss_affine_scan_log_step if log_step else ss.ss_affine_scan
        w, _, _, a, b = affine_setup(torch, dev, name)
        if args.affine_n:
            w = workloads.AffineWorkload(name, args.affine_n, w.a_lo, w.a_hi)
            a, b = a[: w.n].contiguous(), b[: w.n].contiguous()
        h = torch.empty_like(a)
        ws = ss.new_workspace(ss.ss_affine_scan_workspace_bytes(w.n), dev)
        per, _ = time_launches(torch, lambda: fn(a, b, h, workspace=ws, stream=stream),
                               args.steps, args.warmup, stream)
        ms = statistics.mean(per)
        r = {"elements": w.n, "ms": ms, "elements_per_s": w.n / (ms * 1e-3),
             "gbs": 12 * w.n / (ms * 1e-3) / 1e9, "roofline_frac": 12 * w.n / (ms * 1e-3) / 1e9 / hbm_peak}
    else:
        raise SystemExit(f"unknown workload {name}")
    print(json.dumps({"workload": args.workload, "steps": args.steps, "warmup": args.warmup, **r}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="headline workload only")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true",
                    help="skip the oracle timings beside each S6 config")
    ap.add_argument("--affine-n", type=int, default=0,
                    help="with --workload affine_*: use this many elements (small ncu captures)")
    ap.add_argument("--workload", default=HEADLINE,
                    help="time one workload only (affine_small, affine_large, s6_fp32, "
                         "affine_large_log_step, s6_bf16, s6_bidir, s6_bf16_state, s6_fp32_bwd, s6_bf16_bwd, "
                         "s6_bf16_layer, proj_gemm_bf16); "
                         "the default "
                         "is the full benchmark")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.workload != HEADLINE or args.affine_n:
        run_single(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
