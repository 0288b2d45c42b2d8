"""Shared helpers for the GPU parity tests: run libfattn through its C ABI on
seeded workloads and compare with the fp64 oracle.

Tolerances (the ones stated for this method on 16-bit inputs), all raw:
  O    max |O - O_ref|                            <= 1e-2
  LSE  max |LSE - LSE_ref|                        <= 1e-3
  dX   max |dX - dX_ref| / max(max|dX_ref|, 1e-2) <= 2e-2   for X in {Q, K, V}

O is delivered in the inputs' 16-bit type, so rounding the exact O alone
moves it by up to half a unit in the last place (2^-7 for bf16 values in
[2, 4)); the forward's own error must fit in what is left.  check_forward
prints both figures and the rounding floor max |rn16(O_ref) - O_ref|.

Where the exact gradient vanishes everywhere (a single visible key, so the
softmax is constant) the relative bound would be zero; the denominator has a
floor of 1e-2, i.e. an absolute bound of 2e-4 there.
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


def round16(x, dtype):
    """x rounded to the 16-bit type (nearest even), back in float64."""
    t = torch.bfloat16 if dtype == "bf16" else torch.float16
    return torch.from_numpy(np.asarray(x, np.float64)).to(t).double().numpy()


def o_err(got, ref, dtype=None):
    """max |got - ref|: the stated O bound applies to this raw figure."""
    return max_abs(got, ref)


def o_err_beyond_rounding(got, ref, dtype):
    """Diagnostic: max |got - ref| beyond half an output ulp of the exact
    value, i.e. the part of the error the output rounding does not explain."""
    ref = np.asarray(ref, np.float64)
    d = np.abs(np.asarray(got, np.float64) - ref) - half_ulp16(ref, dtype)
    return float(max(np.max(d), 0.0))


def check_forward(w, inputs, o, lse, label=None):
    """Compares O and LSE on the oracle's rows; prints and returns the errors."""
    rows = rows_for(w) if w.sampled else None
    if rows is None:
        ref = oracle_full(w, inputs)
    else:
        ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale, w.causal,
                               rows=rows)
    if rows is not None:
        o_g, lse_g = gather_rows(o, rows), gather_rows(lse, rows)
    else:
        o_g, lse_g = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(np.isfinite(o_g)) and np.all(np.isfinite(lse_g))
    err_o, err_l = o_err(o_g, ref["o"]), max_abs(lse_g, ref["lse"])
    floor = max_abs(round16(ref["o"], w.dtype), ref["o"])
    beyond = o_err_beyond_rounding(o_g, ref["o"], w.dtype)
    print(f"[parity] {label or w.describe()}: O raw {err_o:.3e} (rounding floor {floor:.3e}, "
          f"beyond half an ulp {beyond:.3e}), LSE {err_l:.3e}")
    # the bound is reachable at all: rounding the exact O stays inside it
    assert floor <= TOL_O, f"rounding the exact O alone gives {floor:.3e}"
    assert err_o <= TOL_O, f"O error {err_o:.3e}"
    assert err_l <= TOL_LSE, f"LSE error {err_l:.3e}"
    return err_o, err_l


_full_cache = {}


def oracle_full(w, inputs):
    """The oracle on every row of a workload (with gradients when the inputs
    carry dO).  The last result is kept, so that a forward check and the
    backward checks of both modes on the same inputs run the oracle once."""
    key = (w, "do" in inputs)
    if key not in _full_cache:
        _full_cache.clear()
        _full_cache[key] = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale,
                                            w.causal, dout=inputs.get("do"))
    return _full_cache[key]


def check_backward_full(w, inputs, dq, dk, dv):
    ref = oracle_full(w, inputs)
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
    if w.causal:
        b, h = 0, w.H // 2
        k0, k1 = interior_key_tile(w)
        ref_dk, ref_dv = oracle_key_tile_grads(w, inputs, b, h, k0, k1)
        for name, got, r in (("dk", dk, ref_dk), ("dv", dv, ref_dv)):
            g = got[b, h, k0:k1].float().cpu().numpy()
            errs[name + "_interior"] = rel_err(g, r)
            assert errs[name + "_interior"] <= TOL_GRAD_REL, f"{name} interior tile error"
    errs.update(check_invariants(w, inputs, dk, dv))
    print(f"[parity] {w.describe()} sampled backward: " +
          ", ".join(f"{k} {v:.3e}" for k, v in errs.items()))
    return errs


def interior_key_tile(w, tile=128):
    """Keys [k0, k0 + tile) of one interior key tile, three quarters of the
    way along the sequence."""
    k0 = (3 * w.N // 4) // tile * tile
    return k0, min(k0 + tile, w.N)


_key_tile_cache = {}


def oracle_key_tile_grads(w, inputs, b, h, k0, k1, chunk=1024):
    """Exact dK, dV of keys [k0, k1) of head (b, h).  Each is a column sum
    over every query row that sees those keys (all rows from k0 on under the
    causal mask); the oracle sums over the rows of one call, so the rows are
    taken in chunks and the chunks' sums added."""
    key = (w.name, b, h, k0, k1)
    if key not in _key_tile_cache:
        first = k0 if w.causal else 0
        q, k, v, do = (inputs[n][b, h] for n in ("q", "k", "v", "do"))
        dk = np.zeros((k1 - k0, w.D))
        dv = np.zeros((k1 - k0, w.D))
        for r0 in range(first, w.N, chunk):
            rows = np.arange(r0, min(r0 + chunk, w.N))
            res = oracle.attention_head(q, k, v, w.scale, w.causal, dout=do, rows=rows,
                                        kv_range=(k0, k1))
            dk += res["dk"]
            dv += res["dv"]
        _key_tile_cache[key] = (dk, dv)
    return _key_tile_cache[key]


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
