"""The forward with resident CTAs: short sequences (at most 32 key tiles)
with more work units (pairs of query tiles of one head) than SMs run one
CTA per SM, each walking several units with barrier phases counted across
them.  Checked two ways: against the fp64 oracle on several heads, and bit
for bit against single-head calls of the same inputs, whose few units run
one per CTA.  The arithmetic of a unit does not depend on which CTA runs it
or on what ran before it, so the two launches must agree exactly."""
import numpy as np
import pytest
import torch

import fp8_bound
import oracle
import oracle.fp8 as ofp8
from exact_attention_93_gb300 import fattn, workloads as W

pytestmark = pytest.mark.gpu


def forward(q, k, v, scale, causal, opts=None):
    # NaN-filled outputs: a unit no CTA ran would leave NaN behind
    B, H, N, D = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    fattn.fa_fwd_ex(q, k, v, o, lse, None, opts, B, H, N, D, scale, causal)
    return o, lse


@pytest.mark.parametrize("B,H,N,dtype,causal,window,alibi,seed", [
    (2, 40, 1000, "bf16", True, (-1, -1), False, 61),     # 320 units of 1..8 key tiles
    (1, 100, 777, "fp16", False, (100, 50), True, 62),    # 400 units, window and ALiBi
    (4, 64, 300, "bf16", False, (-1, -1), False, 63),     # 512 units, ragged last tile
    (1, 160, 4096, "bf16", True, (-1, -1), True, 64),     # 32 key tiles, 2560 units
])
def test_resident_forward_matches_oracle_and_single_head_calls(B, H, N, dtype, causal, window,
                                                               alibi, seed):
    w = W.custom(B, H, N, 64, dtype, causal=causal, seed=seed, backward=False)
    inputs = W.make_inputs(w)
    q, k, v = (inputs[n].cuda() for n in "qkv")
    slopes = (torch.linspace(0.02, 0.5, H, dtype=torch.float32) if alibi else None)
    opts = fattn.options(window, slopes.cuda() if alibi else None, None)
    o, lse = forward(q, k, v, w.scale, causal, opts)
    torch.cuda.synchronize()
    assert fattn.fa_device_error() == fattn.FA_OK
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()  # every unit ran
    heads = [(0, 0), (B - 1, H // 2), (B - 1, H - 1)]
    for b, h in heads:
        # the same head alone: one unit per CTA
        sl = None if slopes is None else slopes[h:h + 1].cuda()
        o1, lse1 = forward(q[b:b + 1, h:h + 1].contiguous(), k[b:b + 1, h:h + 1].contiguous(),
                           v[b:b + 1, h:h + 1].contiguous(), w.scale, causal,
                           fattn.options(window, sl, None))
        torch.cuda.synchronize()
        assert torch.equal(o1[0, 0], o[b, h]) and torch.equal(lse1[0, 0], lse[b, h])
        rows = (np.arange(N) if N <= 1000 else
                np.sort(np.random.default_rng(seed + h).choice(N, 96, replace=False)))
        ref = oracle.attention_head(inputs["q"][b, h], inputs["k"][b, h], inputs["v"][b, h],
                                    w.scale, causal, rows=rows, window=window,
                                    alibi_slope=float(slopes[h]) if alibi else 0.0)
        assert np.max(np.abs(o[b, h].float().cpu().numpy()[rows] - ref["o"])) < 1e-2
        assert np.max(np.abs(lse[b, h].cpu().numpy()[rows] - ref["lse"])) < 1e-3


@pytest.mark.parametrize("B,H,N,D,causal,seed", [
    (1, 80, 640, 64, True, 65),     # 240 units
    (2, 90, 300, 128, False, 66),   # 360 units
])
def test_resident_fp8_forward(B, H, N, D, causal, seed):
    d = W.make_fp8_inputs(W.custom(B, H, N, D, causal=causal, seed=seed, backward=False))
    q8, k8, v8 = (d[n].cuda() for n in ("q8", "k8", "v8"))
    desc = [d["descale_" + n].cuda() for n in "qkv"]
    scale = D ** -0.5

    def run(sl_b, sl_h):
        qq, kk, vv = (x[sl_b, sl_h].contiguous() for x in (q8, k8, v8))
        dd = [x[sl_b, sl_h].contiguous() for x in desc]
        b, h = qq.shape[:2]
        o = torch.full((b, h, N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((b, h, N), float("nan"), dtype=torch.float32, device="cuda")
        fattn.fa_fwd_fp8(qq, kk, vv, o, lse, None, None, b, h, N, D, scale, causal, *dd)
        return o, lse

    o, lse = run(slice(None), slice(None))
    torch.cuda.synchronize()
    assert fattn.fa_device_error() == fattn.FA_OK
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()  # every unit ran
    qd, kd, vd = ofp8.dequantise(d["q8"], d["k8"], d["v8"], d["descale_q"], d["descale_k"],
                                 d["descale_v"])
    for b, h in ((0, 0), (B - 1, H - 1)):
        o1, lse1 = run(slice(b, b + 1), slice(h, h + 1))
        torch.cuda.synchronize()
        assert torch.equal(o1[0, 0], o[b, h]) and torch.equal(lse1[0, 0], lse[b, h])
        r = np.arange(N)
        ref = oracle.attention_head(qd[b, h], kd[b, h], vd[b, h], scale, causal, rows=r,
                                    want_probs=True)
        fp8_bound.check_head(o[b, h].float().cpu().numpy(), lse[b, h].cpu().numpy(), ref,
                             qd[b, h], kd[b, h], vd[b, h], scale, r, 0.0, label=f"b{b} h{h}")

