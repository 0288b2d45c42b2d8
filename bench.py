#!/usr/bin/env python3
"""Benchmark: exact attention forward + backward through libfattn on GB300.

One step is the whole path on one batch of seeded synthetic input already in
HBM: fa_fwd, then the backward stages (Di preprocess, dK/dV with atomic dQ,
dQ convert), exactly what fa_bwd enqueues.  The default workload is the
long-sequence causal case B1 H8 N65536 D128 bf16; every input tensor
(134 MB) is larger than the 129 MB L2, so no flush is needed between steps.

Throughput is FLOP/s with the method's own count: 4*B*H*N^2*D for the
forward, 2.5x that for the backward, halved under the causal mask.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed alone

Several GPUs (torchrun, one rank per GPU): every rank runs its own replica
of the workload (independent problems, no data exchange); the value is all
ranks' work over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s fwd and fwd+bwd on 1×GB300; % of dense BF16 tensor peak"
DOMINANT = "bwd_dkdv"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long64k_causal")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the two-pass deterministic backward instead of atomic dQ")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the forward-only long-context measurement")
    ap.add_argument("--fp8-only", action="store_true",
                    help="time only the FP8 forward (fa_fwd_fp8) on e4m3 draws of the workload")
    ap.add_argument("--fwd-only", action="store_true",
                    help="time only the forward (fa_fwd) on the workload")
    return ap.parse_args()


# --------------------------------------------------------------------------
# environment helpers
# --------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    """Measured dense bf16 peaks (TFLOP/s) and HBM GB/s, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"burst": float(d["bf16_tflops"]), "sustained": float(d["bf16_tflops_sustained"]),
                "hbm": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"burst": 1900.0, "sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def code_text(src: str) -> str:
    """C/C++/CUDA source with comments removed and whitespace collapsed: the
    part of a file that decides what the compiler builds."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash(sources: dict | None = None):
    """sha256 prefix over the code of every file in csrc/ (comments and
    whitespace ignored), or of `sources` ({file name: text})."""
    if sources is None:
        d = os.path.join(ROOT, "exact_attention_93_gb300", "csrc")
        sources = {f: open(os.path.join(d, f), encoding="utf-8").read() for f in os.listdir(d)}
    h = hashlib.sha256()
    for name in sorted(sources):
        h.update(name.encode() + b"\0" + code_text(sources[name]).encode() + b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.md")
    if not os.path.exists(p):
        return None
    src = kernel_source_hash()
    for line in open(p):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload:
            try:
                return float(cells[2]) if cells[3] == src else None
            except ValueError:
                return None
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for r in csv.reader(io.StringIO(getattr(self, "out", "") or "")):
            if len(r) >= 9:
                rows.append([x.strip() for x in r])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def slowest_rank(value: float, dist, device) -> float:
    """The largest value over all ranks (the slowest rank's time); the value
    itself on a single process."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank: float, ms_per_step: float) -> float:
    """All ranks' work (each rank runs its own replica) over one step's time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


# --------------------------------------------------------------------------
# the CPU baseline: the fp64 oracle on a bounded sample of the workload
# --------------------------------------------------------------------------

def oracle_sample(w, inputs, rows_per_head):
    """Rows of the workload whose whole forward + backward share the oracle
    computes: O, LSE, dQ for the row and its contributions to dK and dV."""
    import numpy as np
    rows = []
    flops = 0.0
    for h in range(w.H):
        # evenly spaced query rows, so causal rows of every length are timed
        r = np.unique(np.linspace(0, w.N - 1, min(rows_per_head, w.N)).astype(np.int64))
        rows.append(r)
        vis = (r + 1) if w.causal else [w.N] * len(r)
        flops += sum(14.0 * float(v) * w.D for v in vis)  # 4 fwd + 10 bwd per key per dim
    return rows, flops


def time_oracle(w, inputs, rows_per_head):
    import oracle
    oracle.build()
    rows, flops = oracle_sample(w, inputs, rows_per_head)
    t0 = time.perf_counter()
    for h in range(w.H):
        oracle.attention_head(inputs["q"][0, h], inputs["k"][0, h], inputs["v"][0, h], w.scale,
                              w.causal, dout=inputs["do"][0, h], rows=rows[h],
                              kv_range=(0, w.N))
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, sum(len(r) for r in rows), oracle.threads()


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from exact_attention_93_gb300 import workloads as W
    inputs = W.make_inputs(w)
    rows_per_head = 64
    for _ in range(args.warmup):
        time_oracle(w, inputs, 2)
    vals, secs = [], 0.0
    cores = 1
    for _ in range(args.steps):
        v, dt, nrows, cores = time_oracle(w, inputs, rows_per_head)
        vals.append(v)
        secs += dt
    value = statistics.mean(vals)
    sample = (f"{rows_per_head} query rows per head x {w.H} heads of {w.describe()} "
              f"(forward and full backward share of each row), fp64")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.describe() + " fwd+bwd", "parallelism": "none (host cores)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def visible_pairs(N: int, causal: bool, left: int, right: int) -> int:
    """(query, key) pairs the band lets through: query i sees keys
    i - left .. i + right (-1: no bound), and j <= i when causal."""
    import numpy as np
    i = np.arange(N, dtype=np.int64)
    lo = np.zeros(N, np.int64) if left < 0 else np.maximum(i - left, 0)
    hi = np.full(N, N - 1, np.int64) if right < 0 else np.minimum(i + right, N - 1)
    if causal:
        hi = np.minimum(hi, i)
    return int(np.maximum(hi - lo + 1, 0).sum())


def block_pairs(N: int, causal: bool, mask) -> int:
    """(query, key) pairs inside the kept 128 x 128 blocks of `mask`
    ([T, T], shared by every head), under the causal mask when asked."""
    import numpy as np
    T = mask.shape[0]
    size = np.array([min(128, N - 128 * t) for t in range(T)], np.int64)
    full = np.outer(size, size)
    if causal:
        # a diagonal block of s rows keeps s (s + 1) / 2 pairs; blocks above
        # the diagonal keep none
        full = np.tril(full, -1) + np.diag(size * (size + 1) // 2)
    return int((full * (np.asarray(mask) != 0)).sum())


def band_extras(w, g, o, lse, dq, dk, dv, ws, stream, pk, det=False):
    """Forward + backward (the run's dQ mode, whose workspace `ws` is) on the
    benchmark inputs with a sliding window, with ALiBi, and with a random
    block mask keeping half the blocks (and the diagonal), credited with the
    FLOPs of the visible pairs only (4 D per pair forward, 2.5 times that
    backward)."""
    import torch

    from exact_attention_93_gb300 import fattn

    B, H, N, D = w.B, w.H, w.N, w.D
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32,
                          device=g["q"].device)
    import numpy as np

    T = (N + 127) // 128
    rng = np.random.default_rng(0)
    bmask = (rng.random((T, T)) < 0.5).astype(np.uint8)
    np.fill_diagonal(bmask, 1)
    bmask_dev = torch.tensor(bmask, device=g["q"].device)
    out = {}
    for label, window, use_alibi, use_mask in (
            ("sliding window 4096", (4095, 0), False, False),
            ("ALiBi", (-1, -1), True, False),
            ("block-sparse, half the 128 x 128 blocks", (-1, -1), False, True)):
        opts = fattn.options(window, slopes if use_alibi else None,
                             bmask_dev if use_mask else None)

        def one():
            fattn.fa_fwd_ex(g["q"], g["k"], g["v"], o, lse, None, opts, B, H, N, D, w.scale,
                            w.causal)
            fattn.fa_bwd_ex(g["q"], g["k"], g["v"], o, lse, g["do"], dq, dk, dv, None, opts,
                            B, H, N, D, w.scale, w.causal, det, ws)

        for _ in range(3):
            one()
        torch.cuda.synchronize()
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        s0.record(stream)
        for _ in range(reps):
            one()
        e0.record(stream)
        torch.cuda.synchronize()
        ms = s0.elapsed_time(e0) / reps
        pairs = block_pairs(N, w.causal, bmask) if use_mask else visible_pairs(N, w.causal, *window)
        flops = 3.5 * 4.0 * B * H * D * pairs
        tf = flops / (ms * 1e-3) / 1e12
        out[f"{w.describe()} fwd+bwd, {label}"] = {
            "tflops": tf, "ms": ms, "frac_of_peak": tf / pk["sustained"],
            "note": "FLOPs of the visible (query, key) pairs only; fa_fwd_ex + fa_bwd_ex"
                    + (" (deterministic dQ)" if det else " (atomic dQ)")}
    if fattn.fa_device_error() != fattn.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait in the band runs")
    return out


_E4M3_PEAK = {}


def e4m3_gemm_peak(dev, size=8192, seconds=4.0):
    """Dense e4m3 tensor-core throughput measured on this GPU, the
    denominator of the FP8 forward's fraction: cuBLASLt through
    torch._scaled_mm on size^3 (2 size^3 FLOP per call, e4m3 x e4m3 with fp32
    accumulation, bf16 out), best single call of 10 (burst) and the mean over
    back-to-back calls for `seconds` (sustained), like the bf16 peaks the
    driver measures.  Falls back to twice the measured bf16 figures (the
    nominal e4m3 / bf16 ratio) where the call is unavailable."""
    import torch

    if dev in _E4M3_PEAK:
        return _E4M3_PEAK[dev]
    try:
        g = torch.Generator(device="cpu").manual_seed(0)
        a = torch.randn(size, size, generator=g).to(dev).to(torch.float8_e4m3fn)
        bt = torch.randn(size, size, generator=g).to(dev).to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=dev)

        def mm():
            return torch._scaled_mm(a, bt.t(), one, one, out_dtype=torch.bfloat16)

        flop = 2.0 * size ** 3
        for _ in range(3):
            mm()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            mm()
            e0.record()
            torch.cuda.synchronize()
            best = min(best, s0.elapsed_time(e0))
        calls = max(10, int(seconds * 1e3 / best))
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(calls):
            mm()
        e0.record()
        torch.cuda.synchronize()
        sust = s0.elapsed_time(e0) / calls
        r = {"burst": flop / (best * 1e-3) / 1e12, "sustained": flop / (sust * 1e-3) / 1e12,
             "source": f"measured: torch._scaled_mm e4m3 {size}^3, best of 10 (burst) and "
                       f"{calls} back-to-back calls (sustained)"}
        del a, bt
    except Exception as exc:  # no e4m3 GEMM in this torch/cuBLAS build
        pk = peaks()
        r = {"burst": 2.0 * pk["burst"], "sustained": 2.0 * pk["sustained"],
             "source": f"{pk['source']} bf16 x 2 (nominal e4m3 / bf16 ratio; "
                       f"e4m3 GEMM unavailable: {type(exc).__name__})"}
    _E4M3_PEAK[dev] = r
    return r


def fp8_extras(w, dev, stream, pk, reps=10, warmup=3):
    """The FP8 forward (fa_fwd_fp8: the V transpose plus the forward kernel)
    on e4m3 draws of the benchmark shape, against the measured sustained
    e4m3 GEMM peak (e4m3_gemm_peak)."""
    import torch

    from exact_attention_93_gb300 import fattn, workloads as W

    pk8 = e4m3_gemm_peak(dev)
    d = {k: v.to(dev) for k, v in W.make_fp8_inputs(w).items()}
    B, H, N, D = w.B, w.H, w.N, w.D
    o = torch.empty(B, H, N, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    ws = fattn.alloc_fp8_workspace(B, H, N, D, dev)

    def one():
        fattn.fa_fwd_fp8(d["q8"], d["k8"], d["v8"], o, lse, None, None, B, H, N, D, w.scale,
                         w.causal, d["descale_q"], d["descale_k"], d["descale_v"], ws)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(reps):
        one()
    e0.record(stream)
    torch.cuda.synchronize()
    if fattn.fa_device_error() != fattn.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait in the FP8 runs")
    ms = s0.elapsed_time(e0) / reps
    tf = w.fwd_flops() / (ms * 1e-3) / 1e12
    return {f"{w.describe().replace(' bf16', '')} e4m3 fwd": {
        "tflops": tf, "ms": ms, "frac_of_e4m3_peak": tf / pk8["sustained"],
        "peak": pk8["sustained"], "peak_burst": pk8["burst"],
        "peak_source": f"e4m3 sustained, {pk8['source']}",
        "note": "fa_fwd_fp8 (V transpose + forward), O in bf16, per-head descale factors"}}


# exp2 throughput of GB300's special-function unit: ex2.approx.ftz.f32
# measured at 32 lanes per clock per SM by tests/test_unit_rates_gpu.py
# (python -m pytest tests/test_unit_rates_gpu.py -m gpu -s prints the rates)
EX2_PER_CLK_SM = 32


def exp_count(w) -> float:
    """Exponentials one forward evaluates: one per visible (query, key) pair,
    B*H*N^2, halved under the causal mask; the backward evaluates as many
    again when it recomputes P."""
    n = float(w.B) * w.H * w.N * w.N
    return n / 2 if w.causal else n


def sm_count(dev) -> int:
    import torch
    return int(torch.cuda.get_device_properties(dev).multi_processor_count)


def exp_peak(sm_mhz: float, sms: int) -> float:
    return EX2_PER_CLK_SM * sms * sm_mhz * 1e6


def time_calls(fn, reps, warmup, stream):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(reps):
        fn()
    e0.record(stream)
    torch.cuda.synchronize()
    return s0.elapsed_time(e0) / reps


def small_config_extras(dev, stream, pk):
    """Forward and forward + backward (atomic dQ) of the two D = 64
    workloads, B8 H12 N1024 causal bf16 and B32 H16 N512 fp16, whose inputs
    fit in L2 (back-to-back calls)."""
    import torch

    from exact_attention_93_gb300 import fattn, workloads as W

    out = {}
    for name in ("gpt2_causal", "bert_fp16"):
        w = W.WORKLOADS[name]
        g = {k: v.to(dev) for k, v in W.make_inputs(w).items()}
        o = torch.empty_like(g["q"])
        lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        ws = fattn.alloc_workspace(w.B, w.H, w.N, w.D, False, dev)

        def fwd():
            fattn.fa_fwd(g["q"], g["k"], g["v"], o, lse, w.scale, w.causal)

        def step():
            fwd()
            fattn.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], dq, dk, dv, w.scale, w.causal,
                         False, ws)

        ms_f = time_calls(fwd, 50, 5, stream)
        ms_s = time_calls(step, 50, 5, stream)
        tf_f = w.fwd_flops() / (ms_f * 1e-3) / 1e12
        tf_s = (w.fwd_flops() + w.bwd_flops()) / (ms_s * 1e-3) / 1e12
        out[f"{w.describe()} fwd"] = {"tflops": tf_f, "ms": ms_f, "frac_of_peak": tf_f / pk["burst"],
                                      "peak_source": f"{pk['source']} bf16 burst"}
        out[f"{w.describe()} fwd+bwd"] = {
            "tflops": tf_s, "ms": ms_s, "frac_of_peak": tf_s / pk["burst"],
            "peak_source": f"{pk['source']} bf16 burst",
            "note": "fa_fwd + fa_bwd (atomic dQ), back-to-back calls; inputs fit in L2"}
    if fattn.fa_device_error() != fattn.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait in the D = 64 runs")
    return out


def run_fwd_only(args, w):
    """One JSON line for the 16-bit forward alone (profiling and sweeps)."""
    import torch

    from exact_attention_93_gb300 import fattn, workloads as W

    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g = {k: v.to(dev) for k, v in W.make_inputs(w, with_grad_output=False).items()}
    o = torch.empty_like(g["q"])
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    ms = time_calls(lambda: fattn.fa_fwd(g["q"], g["k"], g["v"], o, lse, w.scale, w.causal),
                    args.steps, max(args.warmup, 3), torch.cuda.current_stream())
    if fattn.fa_device_error() != fattn.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait")
    tf = w.fwd_flops() / (ms * 1e-3) / 1e12
    pk = peaks()
    print(json.dumps({"metric": "attention forward TFLOP/s", "value": tf, "unit": "TFLOP/s",
                      "ms": ms, "workload": w.describe(), "frac_of_burst_peak": tf / pk["burst"],
                      "exp_per_s": exp_count(w) / (ms * 1e-3), "steps": args.steps}), flush=True)


def run_fp8_only(args, w):
    """One JSON line for the FP8 forward alone (profiling and sweeps)."""
    import torch

    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    res = fp8_extras(w, dev, torch.cuda.current_stream(), peaks(), reps=args.steps,
                     warmup=max(args.warmup, 3))
    (label, r), = res.items()
    print(json.dumps({"metric": "e4m3 attention forward TFLOP/s", "value": r["tflops"],
                      "unit": "TFLOP/s", "ms": r["ms"], "workload": label,
                      "frac_of_e4m3_peak": r["frac_of_e4m3_peak"], "steps": args.steps}),
          flush=True)


def measure_e2e(args, w, inputs, dev, det, dist, world, flops):
    """The step end to end through the same C-ABI calls, from pinned host
    memory to pinned host memory.  Every step copies its four inputs in and
    its five results (O, LSE, dQ, dK, dV) out inside the timed region; the
    copies run on their own streams, double-buffered, so step k + 1's inputs
    travel while step k computes and step k - 1's results travel back, as a
    prefetching training loop would run them."""
    import torch

    from exact_attention_93_gb300 import fattn

    B, H, N, D = w.B, w.H, w.N, w.D
    pin = {k: v.pin_memory() for k, v in inputs.items()}
    sets = []
    for _ in range(2):
        g = {k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in inputs.items()}
        sets.append({
            "g": g, "o": torch.empty_like(g["q"]),
            "lse": torch.empty(B, H, N, dtype=torch.float32, device=dev),
            "dq": torch.empty_like(g["q"]), "dk": torch.empty_like(g["q"]),
            "dv": torch.empty_like(g["q"]),
            "ws": fattn.alloc_workspace(B, H, N, D, det, dev)})
    out_names = ("o", "lse", "dq", "dk", "dv")
    host_out = [{k: torch.empty(sets[0][k].shape, dtype=sets[0][k].dtype, pin_memory=True)
                 for k in out_names} for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "comp", "out")}

    def compute(S):
        g = S["g"]
        fattn.fa_fwd(g["q"], g["k"], g["v"], S["o"], S["lse"], w.scale, w.causal)
        fattn.fa_bwd(g["q"], g["k"], g["v"], S["o"], S["lse"], g["do"], S["dq"], S["dk"],
                     S["dv"], w.scale, w.causal, det, S["ws"])

    comp_ev = []  # (start, end) of each step's compute on its stream

    def run(steps, start=None, end=None):
        comp_ev.clear()
        if start is not None:
            start.record(s_in)
        for k in range(steps):
            b = k % 2
            S = sets[b]
            if k >= 2:
                s_in.wait_event(ev["comp"][b])  # step k - 2 no longer reads set b's inputs
            with torch.cuda.stream(s_in):
                for name in pin:
                    S["g"][name].copy_(pin[name], non_blocking=True)
                ev["in"][b].record(s_in)
            s_comp.wait_event(ev["in"][b])
            if k >= 2:
                s_comp.wait_event(ev["out"][b])  # step k - 2's results have left set b
            with torch.cuda.stream(s_comp):
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(s_comp)
                compute(S)
                c1.record(s_comp)
                comp_ev.append((c0, c1))
                ev["comp"][b].record(s_comp)
            s_out.wait_event(ev["comp"][b])
            with torch.cuda.stream(s_out):
                for name in out_names:
                    host_out[b][name].copy_(S[name], non_blocking=True)
                ev["out"][b].record(s_out)
        if end is not None:
            end.record(s_out)

    run(2)
    torch.cuda.synchronize()
    if fattn.fa_device_error() != fattn.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait in the end-to-end runs")
    if dist is not None:
        dist.barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(args.steps, s2, e2)
    torch.cuda.synchronize()
    e_ms = slowest_rank(s2.elapsed_time(e2) / args.steps, dist, dev)
    # the compute alone inside that loop (while the copies run beside it)
    comp_ms = statistics.median(a.elapsed_time(b) for a, b in comp_ev)

    # the copies alone, for context (outside the timed region)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s_in):
        t0.record(s_in)
        for name in pin:
            sets[0]["g"][name].copy_(pin[name], non_blocking=True)
        t1.record(s_in)
    torch.cuda.synchronize()
    h2d_ms = t0.elapsed_time(t1)
    with torch.cuda.stream(s_out):
        t0.record(s_out)
        for name in out_names:
            host_out[0][name].copy_(sets[0][name], non_blocking=True)
        t1.record(s_out)
    torch.cuda.synchronize()
    d2h_ms = t0.elapsed_time(t1)
    return {"value": whole_job_tflops(world, flops, e_ms), "unit": "TFLOP/s", "ms_per_step": e_ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbps_alone": h2d / (h2d_ms * 1e-3) / 1e9, "d2h_gbps_alone": d2h / (d2h_ms * 1e-3) / 1e9,
            "compute_ms_per_step_in_loop": comp_ms,
            "pipeline": "copies on their own streams, double-buffered: step k+1's inputs and step "
                        "k-1's results travel while step k computes"}


def run_ours(args, w):
    import torch

    from exact_attention_93_gb300 import fattn, workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fattn.load()

    inputs = W.make_inputs(w)  # every rank runs the same replica
    dev = torch.device("cuda", local)
    g = {k: v.to(dev) for k, v in inputs.items()}
    B, H, N, D = w.B, w.H, w.N, w.D
    o = torch.empty_like(g["q"])
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
    det = bool(args.deterministic)
    ws = fattn.alloc_workspace(B, H, N, D, det, dev)
    stream = torch.cuda.current_stream()

    names = ["fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq" if det else "bwd_dq_convert"]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fattn.fa_fwd(g["q"], g["k"], g["v"], o, lse, w.scale, w.causal)
        if ev is not None:
            ev[1].record(stream)
        fattn.fa_bwd_preprocess(o, g["do"], lse, det, ws)
        if ev is not None:
            ev[2].record(stream)
        fattn.fa_bwd_dkdv(g["q"], g["k"], g["v"], g["do"], dk, dv, w.scale, w.causal, det, ws)
        if ev is not None:
            ev[3].record(stream)
        if det:
            fattn.fa_bwd_dq(g["q"], g["k"], g["v"], g["do"], dq, w.scale, w.causal, ws)
        else:
            fattn.fa_bwd_dq_convert(dq, w.scale, ws)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if fattn.fa_device_error() != fattn.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait during warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # let the sampler start
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(args.steps):
            step(events[k])
        end.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    per_kernel = {n: statistics.mean(ev[i].elapsed_time(ev[i + 1]) for ev in events)
                  for i, n in enumerate(names)}
    if fattn.fa_device_error() != fattn.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait")
    total_ms = slowest_rank(total_ms, dist, dev)

    ms_step = total_ms / args.steps
    fwd_f, bwd_f = w.fwd_flops(), w.bwd_flops()
    bwd_alg = bwd_f  # the deterministic pass's recomputation of S and dP is not credited
    value = whole_job_tflops(world, fwd_f + bwd_alg, ms_step)
    pk = peaks()
    peak_sust = pk["sustained"]
    fwd_tf = fwd_f / (per_kernel["fwd"] * 1e-3) / 1e12
    bwd_ms = sum(per_kernel[n] for n in names[1:])
    bwd_tf = bwd_alg / (bwd_ms * 1e-3) / 1e12

    # dominant kernel: the largest share of the step
    dom = max(per_kernel, key=per_kernel.get)
    # contraction FLOPs each tile kernel performs per launch (each N x N x D
    # contraction is 2*N^2*D per head, halved under the causal mask):
    #   fwd: S, PV (2);  dkdv atomic: S^T, dP^T, dV, dK, dQ (5);  dkdv
    #   deterministic: the first four (4);  dq: S, dP, dQ (3)
    dom_flops = {"fwd": fwd_f, "bwd_dkdv": (0.8 if det else 1.0) * bwd_f,
                 "bwd_dq": 0.6 * bwd_f}.get(dom)
    if dom_flops is not None:
        achieved = dom_flops / (per_kernel[dom] * 1e-3) / 1e12
        # the deterministic dK/dV kernel (no dQ) is another kernel with its own traffic
        traffic_key = "bwd_dkdv_deterministic" if det and dom == "bwd_dkdv" else dom
        roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak_sust,
                    "unit": "TFLOP/s", "frac": achieved / peak_sust,
                    "peak_source": f"{pk['source']} bf16 sustained",
                    "traffic": recorded_traffic(traffic_key, w.name),
                    # the sources the traffic row (profiles/dram_traffic.md) must match
                    "kernel_sources": kernel_source_hash()}
    else:  # an elementwise kernel dominating would be HBM bound
        roofline = {"kernel": dom, "bound": "hbm", "achieved": None, "peak": pk["hbm"],
                    "unit": "GB/s", "frac": None, "traffic": None}

    # end to end through the C ABI with host buffers: H2D inputs, step, D2H results
    e2e = None
    if not args.no_e2e:
        with ClockSampler(local) as clk_e2e:
            e2e = measure_e2e(args, w, inputs, dev, det, dist, world, fwd_f + bwd_alg)
        # the clocks while copies and compute overlap (power draw is higher)
        e2e["clocks"] = clk_e2e.summary()

    # the long-context forward-only workload, reported beside the step
    extra = {}
    if rank == 0 and w.name == "long64k_causal" and not args.no_extra:
        w2 = W.WORKLOADS["long4k_fwd"]
        i2 = {k: v.to(dev) for k, v in W.make_inputs(w2).items()}
        o2 = torch.empty_like(i2["q"])
        l2 = torch.empty(w2.B, w2.H, w2.N, dtype=torch.float32, device=dev)
        for _ in range(5):
            fattn.fa_fwd(i2["q"], i2["k"], i2["v"], o2, l2, w2.scale, w2.causal)
        torch.cuda.synchronize()
        s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 50
        s3.record(stream)
        for _ in range(reps):
            fattn.fa_fwd(i2["q"], i2["k"], i2["v"], o2, l2, w2.scale, w2.causal)
        e3.record(stream)
        torch.cuda.synchronize()
        ms2 = s3.elapsed_time(e3) / reps
        tf2 = w2.fwd_flops() / (ms2 * 1e-3) / 1e12
        extra[w2.describe() + " fwd"] = {"tflops": tf2, "ms": ms2,
                                         "frac_of_burst_peak": tf2 / pk["burst"],
                                         "note": "back-to-back launches; inputs 16.8 MB each fit in L2"}
        extra.update(band_extras(w, g, o, lse, dq, dk, dv, ws, stream, pk, det))
        extra.update(fp8_extras(w, dev, stream, pk))
        # head dimension 64 at the same sequence length and work (twice the heads)
        extra.update(fp8_extras(W.custom(w.B, 2 * w.H, w.N, 64, causal=w.causal, seed=w.seed,
                                         backward=False), dev, stream, pk))
        extra.update(small_config_extras(dev, stream, pk))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, nrows, cores = time_oracle(w, inputs, 1024)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{nrows} query rows of {w.describe()} ({nrows // w.H} per head), "
                         f"each row's whole forward and backward share, fp64, {dt:.1f} s"}

    # the secondary ceiling: exponentials per second against the unit's rate
    clk_summary = clk.summary()
    mhz = clk_summary.get("sm_mhz") or 2070.0
    n_exp = exp_count(w)
    exp_rate = {"fwd": n_exp / (per_kernel["fwd"] * 1e-3),
                "bwd_dkdv": n_exp / (per_kernel["bwd_dkdv"] * 1e-3),
                "unit": "exp/s", "peak": exp_peak(mhz, sm_count(dev)),
                "peak_source": f"{EX2_PER_CLK_SM} ex2 lanes/clk/SM (measured) x "
                               f"{sm_count(dev)} SMs x {mhz:.0f} MHz"}
    exp_rate["frac_fwd"] = exp_rate["fwd"] / exp_rate["peak"]

    launches = len(names) * args.steps  # one kernel per entry-point call
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": f"{w.describe()} fwd+bwd "
                                   f"({'deterministic two-pass dQ' if det else 'atomic dQ'})",
                       "B": B, "H": H, "N": N, "D": D, "causal": w.causal,
                       "l2": (f"inputs larger than L2 (each input tensor "
                              f"{B * H * N * D * 2 / 1e6:.0f} MB > 129 MB), no flush"
                              if B * H * N * D * 2 > 129e6 else
                              f"inputs fit in L2 (each input tensor "
                              f"{B * H * N * D * 2 / 1e6:.0f} MB), no flush: a warm-L2 figure"),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "frac_of_peak": {"fwd+bwd": value / world / peak_sust, "fwd": fwd_tf / peak_sust,
                             "peak": peak_sust, "peak_source": f"{pk['source']} bf16 sustained"},
            "kernel_ms": per_kernel,
            "exp_rate": exp_rate,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk_summary,
            "extra": extra,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    from exact_attention_93_gb300 import workloads as W
    if args.workload.startswith("custom:"):
        B, H, N, D, dt, c = args.workload.split(":", 1)[1].split(",")
        w = W.custom(int(B), int(H), int(N), int(D), dtype=dt, causal=c in ("1", "causal"),
                     seed=4)
    else:
        w = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        if not w.backward:
            raise SystemExit(f"workload {args.workload} has no backward; pick one that does")
        run_reference(args, w)
    elif args.fp8_only:
        run_fp8_only(args, w)
    elif args.fwd_only:
        run_fwd_only(args, w)
    elif not w.backward:
        raise SystemExit(f"workload {args.workload} has no backward; use --fwd-only")
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
