"""Sliding-window attention and ALiBi on the GPU against the fp64 oracle.

flash_attn_func's window_size = (left, right) lets query i see keys
i - left .. i + right (-1: no bound) and alibi_slopes adds -slope * |i - j|
to the score (claire-chang.com FlashAttention introduction).  Windows are
chosen to fall inside one 128-key tile, to span several, to be one-sided
and to meet the causal mask; every case runs the forward and both backward
modes through fa_fwd_ex / fa_bwd_ex and is checked element by element."""
import numpy as np
import pytest
import torch

import oracle
import parity_util as U
from exact_attention_93_gb300 import fattn, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fattn.load()
    yield
    U.assert_no_device_error()


def alibi(B, H, per_batch):
    """Geometric slopes 2^(-8 (h + 1) / H), varied per batch when asked."""
    s = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)])
    if per_batch:
        s = np.stack([s * (1.0 + 0.5 * b) for b in range(B)])
    return s.astype(np.float32)


def run_and_check(B, H, N, D, dtype, causal, window, slopes=None, modes=(False, True)):
    w = W.custom(B, H, N, D, dtype=dtype, causal=causal, seed=N * 3 + D + window[0] % 7)
    inputs = W.make_inputs(w)
    g = U.gpu_inputs(w, inputs)
    sl = torch.tensor(slopes, device="cuda") if slopes is not None else None
    opts = fattn.options(window, sl)
    o = torch.empty_like(g["q"])
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    fattn.fa_fwd_ex(g["q"], g["k"], g["v"], o, lse, None, opts, B, H, N, D, w.scale, causal)
    torch.cuda.synchronize()
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale, causal,
                           dout=inputs["do"], window=window, alibi_slopes=slopes)
    err_o = U.o_err(o.float().cpu().numpy(), ref["o"], dtype)
    print(f"[parity] {w.describe()} window {window} alibi {slopes is not None}: O raw {err_o:.3e}")
    err_l = U.max_abs(lse.cpu().numpy(), ref["lse"])
    assert err_o <= U.TOL_O, f"O error {err_o:.3e}"
    assert err_l <= U.TOL_LSE, f"LSE error {err_l:.3e}"
    for det in modes:
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        fattn.fa_bwd_ex(g["q"], g["k"], g["v"], o, lse, g["do"], dq, dk, dv, None, opts,
                        B, H, N, D, w.scale, causal, det)
        torch.cuda.synchronize()
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            e = U.rel_err(got.float().cpu().numpy(), ref[name])
            assert e <= U.TOL_GRAD_REL, f"{name} ({'det' if det else 'atomic'}) error {e:.3e}"
    U.assert_no_device_error()


WINDOWS = [
    # (B, H, N, D, dtype, causal, (left, right))
    (1, 2, 300, 64, "bf16", False, (32, 16)),      # inside one tile
    (1, 2, 300, 64, "bf16", False, (0, 0)),        # the identity map
    (1, 2, 300, 64, "bf16", True, (127, -1)),      # causal, left-bounded
    (1, 2, 300, 64, "bf16", False, (-1, 64)),      # right-bounded only
    (1, 2, 300, 64, "bf16", False, (200, -1)),     # left-bounded only, spans tiles
    (2, 1, 257, 64, "fp16", False, (16, 300)),
    (1, 2, 400, 128, "bf16", False, (64, 64)),
    (1, 2, 400, 128, "bf16", True, (100, 7)),      # causal ignores the right bound
    (1, 1, 385, 128, "fp16", False, (0, 129)),
    (1, 2, 1024, 128, "bf16", True, (300, 0)),     # several tiles each side
]


@pytest.mark.parametrize("B,H,N,D,dtype,causal,window", WINDOWS)
def test_window_matches_oracle(B, H, N, D, dtype, causal, window):
    run_and_check(B, H, N, D, dtype, causal, window)


RESIDENT = [
    # More (batch, head, key tile) units than SMs at D = 64 and short N: the
    # dK / dV kernel runs resident CTAs that take several units each, with
    # ragged last key tiles and, under the identity window, one-tile units.
    # (B, H, N, D, dtype, causal, (left, right), ALiBi)
    (4, 40, 300, 64, "bf16", False, (32, 16), False),
    (4, 40, 300, 64, "bf16", False, (0, 0), False),
    (2, 80, 200, 64, "fp16", True, (-1, -1), True),
]


@pytest.mark.parametrize("B,H,N,D,dtype,causal,window,use_alibi", RESIDENT)
def test_resident_units_match_oracle(B, H, N, D, dtype, causal, window, use_alibi):
    run_and_check(B, H, N, D, dtype, causal, window, alibi(B, H, True) if use_alibi else None)


ALIBI = [
    # (B, H, N, D, dtype, causal, window, per_batch)
    (2, 3, 257, 64, "bf16", False, (-1, -1), False),
    (2, 3, 257, 64, "bf16", True, (-1, -1), True),
    (1, 2, 300, 128, "fp16", False, (-1, -1), False),
    (2, 2, 200, 128, "bf16", True, (-1, -1), True),
    (1, 2, 400, 128, "bf16", False, (90, 40), False),
    (1, 2, 300, 64, "bf16", True, (64, -1), True),
    # long rows: most tiles lie wholly on one side of the diagonal, where the
    # kernels add the bias in its linear form, over distances up to N - 1
    (1, 2, 2048, 64, "bf16", False, (-1, -1), False),
    (1, 1, 1536, 128, "bf16", True, (-1, -1), False),
]


@pytest.mark.parametrize("B,H,N,D,dtype,causal,window,per_batch", ALIBI)
def test_alibi_matches_oracle(B, H, N, D, dtype, causal, window, per_batch):
    run_and_check(B, H, N, D, dtype, causal, window, alibi(B, H, per_batch))


def test_full_window_is_bitwise_the_plain_call():
    """window (-1, -1) without slopes runs the same code as fa_fwd / fa_bwd."""
    B, H, N, D = 1, 2, 300, 128
    w = W.custom(B, H, N, D, causal=True, seed=17)
    g = U.gpu_inputs(w, W.make_inputs(w))
    o, lse = U.run_forward(w, g)
    dq, dk, dv = U.run_backward(w, g, o, lse, True)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    opts = fattn.options((-1, -1))
    fattn.fa_fwd_ex(g["q"], g["k"], g["v"], o2, lse2, None, opts, B, H, N, D, w.scale, True)
    g2 = [torch.empty_like(dq) for _ in range(3)]
    fattn.fa_bwd_ex(g["q"], g["k"], g["v"], o2, lse2, g["do"], *g2, None, opts, B, H, N, D,
                    w.scale, True, True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    for a, b in zip((dq, dk, dv), g2):
        assert torch.equal(a, b)


def test_window_through_flash_attn_func_autograd():
    from exact_attention_93_gb300.attention import flash_attn_func
    B, H, N, D = 2, 2, 300, 64
    w = W.custom(B, H, N, D, causal=True, seed=19)
    inputs = W.make_inputs(w)
    slopes = alibi(B, H, False)
    q, k, v, do = (inputs[x].cuda().transpose(1, 2).contiguous() for x in ("q", "k", "v", "do"))
    for t in (q, k, v):
        t.requires_grad_()
    o = flash_attn_func(q, k, v, causal=True, window_size=(50, -1),
                        alibi_slopes=torch.tensor(slopes, device="cuda"))
    o.backward(do)
    torch.cuda.synchronize()
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], D ** -0.5, True,
                           dout=inputs["do"], window=(50, -1), alibi_slopes=slopes)
    assert U.o_err(o.detach().transpose(1, 2).float().cpu().numpy(), ref["o"], "bf16") <= U.TOL_O
    for t, name in ((q, "dq"), (k, "dk"), (v, "dv")):
        e = U.rel_err(t.grad.transpose(1, 2).float().cpu().numpy(), ref[name])
        assert e <= U.TOL_GRAD_REL, f"{name} {e:.3e}"
