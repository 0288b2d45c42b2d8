"""Strided layouts, packed QKV and the autograd entry points on the GPU.

The kernels do the same arithmetic whatever the operands' strides, so a
call on (batch, seqlen, nheads, headdim) tensors, or on any mix of layouts,
must reproduce the contiguous call bit for bit: the forward, the
deterministic backward, and dK/dV of the atomic backward (whose dQ sums
fp32 atomics in a run-dependent order).  The autograd entry points are
checked against the fp64 oracle like every other path."""
import pytest
import torch

import oracle
import parity_util as U
from exact_attention_93_gb300 import fattn, workloads as W
from exact_attention_93_gb300.attention import flash_attn_func, flash_attn_qkvpacked_func

pytestmark = pytest.mark.gpu

SHAPES = [
    # (B, H, N, D, dtype, causal): ragged tails, both head sizes, both dtypes
    (2, 3, 200, 64, "bf16", True),
    (1, 2, 256, 128, "fp16", False),
    (2, 2, 129, 128, "bf16", True),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fattn.load()
    yield
    U.assert_no_device_error()


def bnhd(t):
    """A contiguous (B, N, H, D) copy of a [B, H, N, D] tensor."""
    return t.transpose(1, 2).contiguous()


def bhnd_view(t):
    """A (B, N, H, D) tensor seen as [B, H, N, D] (a view, no copy)."""
    return t.transpose(1, 2)


def layout(*ts):
    return fattn.FaLayout(*(fattn.strides_of(t, "bnhd") for t in ts))


def contiguous_reference(w, g, deterministic):
    o, lse = U.run_forward(w, g)
    dq, dk, dv = U.run_backward(w, g, o, lse, deterministic)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("B,H,N,D,dtype,causal", SHAPES)
def test_bnhd_layout_is_bitwise_equal_to_contiguous(B, H, N, D, dtype, causal):
    w = W.custom(B, H, N, D, dtype=dtype, causal=causal, seed=7 + N)
    g = U.gpu_inputs(w, W.make_inputs(w))
    q, k, v, do = (bnhd(g[x]) for x in ("q", "k", "v", "do"))
    for det in (True, False):
        o_c, lse_c, dq_c, dk_c, dv_c = contiguous_reference(w, g, det)
        o, lse = torch.empty_like(q), torch.empty_like(lse_c)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        L = layout(q, k, v, o, do, dq, dk, dv)
        fattn.fa_fwd_strided(q, k, v, o, lse, L, B, H, N, D, w.scale, causal)
        fattn.fa_bwd_strided(q, k, v, o, lse, do, dq, dk, dv, L, B, H, N, D, w.scale, causal, det)
        torch.cuda.synchronize()
        assert torch.equal(bhnd_view(o), o_c) and torch.equal(lse, lse_c)
        assert torch.equal(bhnd_view(dk), dk_c) and torch.equal(bhnd_view(dv), dv_c)
        if det:
            assert torch.equal(bhnd_view(dq), dq_c)
        else:
            assert U.rel_err(bhnd_view(dq).float().cpu().numpy(), dq_c.float().cpu().numpy()) < 1e-2
    U.assert_no_device_error()


def test_mixed_layouts_in_one_call():
    """Each operand in its own layout: Q (B,N,H,D), K contiguous, V inside a
    packed (B,N,3,H,D) buffer, O and the gradients (B,N,H,D), dO a
    transposed view."""
    B, H, N, D = 2, 2, 200, 64
    w = W.custom(B, H, N, D, causal=True, seed=11)
    g = U.gpu_inputs(w, W.make_inputs(w))
    o_c, lse_c, dq_c, dk_c, dv_c = contiguous_reference(w, g, True)
    q = bnhd(g["q"])
    k = g["k"]                                        # [B, H, N, D]
    packed = torch.zeros(B, N, 3, H, D, dtype=g["v"].dtype, device="cuda")
    packed[:, :, 2] = bnhd(g["v"])
    v = packed[:, :, 2]
    do = bnhd(g["do"])                                # (B, N, H, D)
    o = torch.empty_like(q)
    lse = torch.empty_like(lse_c)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    L = fattn.FaLayout(fattn.strides_of(q, "bnhd"), fattn.strides_of(k, "bhnd"),
                       fattn.strides_of(v, "bnhd"), fattn.strides_of(o, "bnhd"),
                       fattn.strides_of(do, "bnhd"), fattn.strides_of(dq, "bnhd"),
                       fattn.strides_of(dk, "bnhd"), fattn.strides_of(dv, "bnhd"))
    fattn.fa_fwd_strided(q, k, v, o, lse, L, B, H, N, D, w.scale, True)
    fattn.fa_bwd_strided(q, k, v, o, lse, do, dq, dk, dv, L, B, H, N, D, w.scale, True, True)
    torch.cuda.synchronize()
    assert torch.equal(bhnd_view(o), o_c) and torch.equal(lse, lse_c)
    for got, ref in ((dq, dq_c), (dk, dk_c), (dv, dv_c)):
        assert torch.equal(bhnd_view(got), ref)
    U.assert_no_device_error()


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "deterministic"])
@pytest.mark.parametrize("causal", [False, True])
def test_flash_attn_func_autograd_matches_oracle(causal, deterministic):
    B, H, N, D = 2, 2, 300, 128
    w = W.custom(B, H, N, D, causal=causal, seed=3)
    inputs = W.make_inputs(w)
    q, k, v, do = (bnhd(inputs[x].cuda()) for x in ("q", "k", "v", "do"))
    for t in (q, k, v):
        t.requires_grad_()
    o = flash_attn_func(q, k, v, causal=causal, deterministic=deterministic)  # default 1/sqrt(D)
    o.backward(do)
    torch.cuda.synchronize()
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], D ** -0.5, causal,
                           dout=inputs["do"])
    assert U.o_err(bhnd_view(o.detach()).float().cpu().numpy(), ref["o"], w.dtype) <= U.TOL_O
    for t, name in ((q, "dq"), (k, "dk"), (v, "dv")):
        e = U.rel_err(bhnd_view(t.grad).float().cpu().numpy(), ref[name])
        assert e <= U.TOL_GRAD_REL, f"{name} relative error {e:.3e}"
    U.assert_no_device_error()


def test_flash_attn_func_returns_the_log_sum_exp():
    B, H, N, D = 1, 2, 200, 64
    w = W.custom(B, H, N, D, causal=True, seed=5)
    inputs = W.make_inputs(w, with_grad_output=False)
    q, k, v = (bnhd(inputs[x].cuda()) for x in ("q", "k", "v"))
    o, lse = flash_attn_func(q, k, v, softmax_scale=0.3, causal=True, return_lse=True)
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], 0.3, True)
    assert lse.shape == (B, H, N)
    assert U.max_abs(lse.cpu().numpy(), ref["lse"]) <= U.TOL_LSE


@pytest.mark.parametrize("causal", [False, True])
def test_qkvpacked_equals_separate_tensors(causal):
    B, H, N, D = 2, 3, 257, 64
    w = W.custom(B, H, N, D, causal=causal, seed=9)
    g = U.gpu_inputs(w, W.make_inputs(w))
    q, k, v, do = (bnhd(g[x]) for x in ("q", "k", "v", "do"))
    qkv = torch.stack([q, k, v], dim=2).requires_grad_()         # (B, N, 3, H, D)
    o_p = flash_attn_qkvpacked_func(qkv, causal=causal, deterministic=True)
    o_p.backward(do)
    qs, ks, vs = (t.clone().requires_grad_() for t in (q, k, v))
    o_s = flash_attn_func(qs, ks, vs, causal=causal, deterministic=True)
    o_s.backward(do)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_s)
    assert qkv.grad.shape == qkv.shape
    for i, t in enumerate((qs, ks, vs)):
        assert torch.equal(qkv.grad[:, :, i], t.grad)
    U.assert_no_device_error()


def test_gradient_in_another_layout_is_used_in_place():
    """An incoming gradient that is a transposed view (D still contiguous)
    goes to the kernels as it is and gives the same result as a copy."""
    B, H, N, D = 1, 2, 200, 64
    w = W.custom(B, H, N, D, causal=True, seed=13)
    g = U.gpu_inputs(w, W.make_inputs(w))
    q, k, v = (bnhd(g[x]).requires_grad_() for x in ("q", "k", "v"))
    do_view = g["do"].transpose(1, 2)                               # (B, N, H, D) view
    assert not do_view.is_contiguous()
    flash_attn_func(q, k, v, causal=True, deterministic=True).backward(do_view)
    grads_view = [t.grad.clone() for t in (q, k, v)]
    for t in (q, k, v):
        t.grad = None
    flash_attn_func(q, k, v, causal=True, deterministic=True).backward(do_view.contiguous())
    for a, t in zip(grads_view, (q, k, v)):
        assert torch.equal(a, t.grad)
