"""Seeded synthetic workloads for exact attention.

This module only draws inputs.  It holds none of the attention arithmetic, so
both the CUDA path and the fp64 oracle can take their inputs from it.

The five workloads are the shapes quoted for the method: a tiny parity case,
a long-context forward (B2 H8 N4096 D128), GPT-2-small-shaped causal
attention (B8 H12 N1024 D64), BERT-large-shaped fp16 attention
(B32 H16 N512 D64) and a long-sequence causal case (B1 H8 N65536 D128).
They stand in for the pages' training workloads (BERT-large at sequence 512,
GPT-2 at 1K, Long-Range Arena at 1K-4K, Path-256 at 64K) by shape only; no
dataset or model is involved.

Drawing rule: one CPU ``torch.Generator`` seeded with the workload's seed;
Q, K, V and then dO are drawn in that order, each as
``torch.randn(B, H, N, D, dtype=float32)``, then rounded to the workload dtype
(round to nearest even).  The fp16 workload scales dO by 0.1 (standard
deviation 0.1) before rounding.  Workloads without a backward draw Q, K, V only.

Query rows checked on large shapes: per (b, h), 256 distinct interior rows
drawn by ``numpy.random.default_rng(seed * 1_000_003 + b * H + h).choice(
arange(1, N - 1), 256, replace=False)``, plus rows 0 and N - 1, sorted (258
rows in all).  For causal workloads the
last key tile's gradient is checked too, which needs the last ``tail`` query
rows in full (see ``tail_rows``).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str          # "bf16" or "fp16"
    causal: bool
    seed: int
    backward: bool
    do_std: float = 1.0
    sampled: bool = False   # oracle checked on sampled rows only

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "fp16": torch.float16}[self.dtype]

    def fwd_flops(self) -> float:
        """4 B H N^2 D, halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.D
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        """2.5 x the forward count (five N x N x D contractions)."""
        return 2.5 * self.fwd_flops()

    def describe(self) -> str:
        return (f"B{self.B} H{self.H} N{self.N} D{self.D} {self.dtype}"
                f"{' causal' if self.causal else ''}")


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 128, 64, "bf16", False, 0, True),
    "long4k_fwd": Workload("long4k_fwd", 2, 8, 4096, 128, "bf16", False, 1,
                           False, sampled=True),
    "gpt2_causal": Workload("gpt2_causal", 8, 12, 1024, 64, "bf16", True, 2, True),
    "bert_fp16": Workload("bert_fp16", 32, 16, 512, 64, "fp16", False, 3, True,
                          do_std=0.1),
    "long64k_causal": Workload("long64k_causal", 1, 8, 65536, 128, "bf16", True,
                               4, True, sampled=True),
}

ORDER = ["tiny", "long4k_fwd", "gpt2_causal", "bert_fp16", "long64k_causal"]


def make_inputs(w: Workload, with_grad_output: bool | None = None):
    """Seeded CPU tensors q, k, v (and do when the workload has a backward)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.D)
    out = {}
    for name in ("q", "k", "v"):
        out[name] = torch.randn(shape, dtype=torch.float32, generator=g).to(w.torch_dtype)
    want = w.backward if with_grad_output is None else with_grad_output
    if want:
        d = torch.randn(shape, dtype=torch.float32, generator=g)
        if w.do_std != 1.0:
            d = d * w.do_std
        out["do"] = d.to(w.torch_dtype)
    return out


E4M3_MAX = 448.0  # largest finite e4m3 value


def make_fp8_inputs(w: Workload):
    """Seeded e4m3 inputs for the FP8 forward: Q, K, V drawn exactly as
    ``make_inputs`` draws them (float32 standard normals, same generator and
    order), then scaled per (b, h) so that the largest magnitude maps to 448
    and rounded to torch.float8_e4m3fn (round to nearest even).  Returns CPU
    tensors q8, k8, v8 [B, H, N, D] and the float32 [B, H] factors
    descale_q, descale_k, descale_v (amax / 448) that map the bytes back to
    the drawn scale."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.D)
    out = {}
    for name in ("q", "k", "v"):
        x = torch.randn(shape, dtype=torch.float32, generator=g)
        amax = x.abs().amax(dim=(2, 3)).clamp_min(1e-30)
        descale = (amax / E4M3_MAX).to(torch.float32)
        out[name + "8"] = (x / descale[:, :, None, None]).to(torch.float8_e4m3fn)
        out["descale_" + name] = descale.contiguous()
    return out


def custom(B, H, N, D, dtype="bf16", causal=False, seed=0, backward=True,
           do_std=1.0) -> Workload:
    """A workload of any shape (edge cases in the tests)."""
    return Workload(f"B{B}H{H}N{N}D{D}{dtype}{'c' if causal else ''}s{seed}",
                    B, H, N, D, dtype, causal, seed, backward, do_std)


def sampled_rows(w: Workload, b: int, h: int, count: int = 256) -> np.ndarray:
    """Sorted distinct query rows checked against the oracle for (b, h)."""
    if not w.sampled or w.N <= count + 2:
        return np.arange(w.N, dtype=np.int64)
    rng = np.random.default_rng(w.seed * 1_000_003 + b * w.H + h)
    r = rng.choice(np.arange(1, w.N - 1), count, replace=False)
    r = np.concatenate([r, np.array([0, w.N - 1])])
    return np.sort(r).astype(np.int64)


def tail_rows(w: Workload, tail: int = 128) -> np.ndarray:
    """The last ``tail`` query rows.  Under the causal mask the keys in
    [N - tail, N) are seen only by these rows, so their dK and dV are exact
    sums over these rows."""
    t = min(tail, w.N)
    return np.arange(w.N - t, w.N, dtype=np.int64)
