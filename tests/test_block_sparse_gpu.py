"""Block-sparse attention on the GPU against the fp64 oracle.

A byte mask over blocks of 128 x 128 scores decides which (query tile, key
tile) pairs are multiplied at all (the block-sparse extension of the
FlashAttention paper that the pages report); the kernels skip the other
tiles.  Masks are random (so query tiles of a pair differ, streams have
gaps, and some tiles are left with nothing), per call or per head, and
combined with the causal mask, a window and ALiBi.  Rows that see no key
must give O = 0, LSE = -inf and no gradient."""
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


def random_mask(T, seed, density=0.5, heads=None, keep_diagonal=False):
    rng = np.random.default_rng(seed)
    shape = (T, T) if heads is None else (heads, T, T)
    m = (rng.random(shape) < density).astype(np.uint8)
    if keep_diagonal:
        idx = np.arange(T)
        if heads is None:
            m[idx, idx] = 1
        else:
            m[:, idx, idx] = 1
    return m


def check_lse(got, ref):
    got = np.asarray(got, np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "rows without keys differ"
    fin = np.isfinite(ref)
    assert U.max_abs(got[fin], ref[fin]) <= U.TOL_LSE


def run_and_check(B, H, N, D, dtype, causal, mask, window=(-1, -1), slopes=None,
                  modes=(False, True)):
    w = W.custom(B, H, N, D, dtype=dtype, causal=causal, seed=int(mask.sum()) + N)
    inputs = W.make_inputs(w)
    g = U.gpu_inputs(w, inputs)
    m_dev = torch.tensor(mask, device="cuda")
    sl = torch.tensor(slopes, device="cuda") if slopes is not None else None
    opts = fattn.options(window, sl, m_dev)
    o = torch.empty_like(g["q"])
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    fattn.fa_fwd_ex(g["q"], g["k"], g["v"], o, lse, None, opts, B, H, N, D, w.scale, causal)
    torch.cuda.synchronize()
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale, causal,
                           dout=inputs["do"], window=window, alibi_slopes=slopes,
                           block_mask=mask, block=128)
    err_o = U.o_err(o.float().cpu().numpy(), ref["o"], dtype)
    print(f"[parity] {w.describe()} block mask, window {window} alibi {slopes is not None}: O raw {err_o:.3e}")
    assert err_o <= U.TOL_O, f"O error {err_o:.3e}"
    check_lse(lse.cpu().numpy(), ref["lse"])
    for det in modes:
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        fattn.fa_bwd_ex(g["q"], g["k"], g["v"], o, lse, g["do"], dq, dk, dv, None, opts,
                        B, H, N, D, w.scale, causal, det)
        torch.cuda.synchronize()
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            e = U.rel_err(got.float().cpu().numpy(), ref[name])
            assert e <= U.TOL_GRAD_REL, f"{name} ({'det' if det else 'atomic'}) error {e:.3e}"
    U.assert_no_device_error()
    return o, lse


CASES = [
    # (B, H, N, D, dtype, causal, seed, density, per_head, keep_diagonal)
    (1, 2, 1000, 64, "bf16", False, 1, 0.5, False, False),
    (1, 2, 1000, 128, "bf16", True, 2, 0.5, False, True),
    (2, 2, 777, 128, "fp16", False, 3, 0.4, True, False),
    (1, 3, 1024, 64, "fp16", True, 4, 0.6, True, False),
    (1, 1, 1300, 128, "bf16", False, 5, 0.25, False, False),
]


@pytest.mark.parametrize("B,H,N,D,dtype,causal,seed,density,per_head,keep_diag", CASES)
def test_random_block_masks_match_oracle(B, H, N, D, dtype, causal, seed, density, per_head,
                                         keep_diag):
    T = (N + 127) // 128
    mask = random_mask(T, seed, density, H if per_head else None, keep_diag)
    run_and_check(B, H, N, D, dtype, causal, mask)


@pytest.mark.parametrize("D", [64, 128])
def test_empty_query_and_key_blocks(D):
    """Block row 2 and block column 5 emptied: those query rows get O = 0 and
    LSE = -inf, those keys get dK = dV = 0."""
    N, T = 1000, 8
    mask = np.ones((T, T), np.uint8)
    mask[2, :] = 0
    mask[:, 5] = 0
    o, lse = run_and_check(1, 2, N, D, "bf16", False, mask)
    assert torch.all(o[:, :, 256:384] == 0)
    assert torch.all(torch.isneginf(lse[:, :, 256:384]))


def test_empty_mask_gives_zeros():
    N, T = 300, 3
    w = W.custom(1, 2, N, 64, seed=21)
    g = U.gpu_inputs(w, W.make_inputs(w))
    opts = fattn.options(block_mask=torch.zeros(T, T, dtype=torch.uint8, device="cuda"))
    o = torch.full_like(g["q"], 7.0)
    lse = torch.zeros(1, 2, N, device="cuda")
    fattn.fa_fwd_ex(g["q"], g["k"], g["v"], o, lse, None, opts, 1, 2, N, 64, w.scale, False)
    for det in (False, True):
        grads = [torch.full_like(g["q"], 7.0) for _ in range(3)]
        fattn.fa_bwd_ex(g["q"], g["k"], g["v"], o, lse, g["do"], *grads, None, opts, 1, 2, N, 64,
                        w.scale, False, det)
        torch.cuda.synchronize()
        for t in grads:
            assert torch.all(t == 0)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    U.assert_no_device_error()


def test_block_mask_with_window_and_alibi():
    N, H, T = 1000, 2, 8
    mask = random_mask(T, 9, 0.6)
    slopes = np.array([0.05, 0.2], np.float32)
    run_and_check(1, H, N, 128, "bf16", True, mask, window=(300, -1), slopes=slopes)


def test_all_ones_mask_is_bitwise_the_dense_call():
    B, H, N, D = 1, 2, 700, 128
    w = W.custom(B, H, N, D, causal=True, seed=23)
    g = U.gpu_inputs(w, W.make_inputs(w))
    o, lse = U.run_forward(w, g)
    dq, dk, dv = U.run_backward(w, g, o, lse, True)
    T = (N + 127) // 128
    opts = fattn.options(block_mask=torch.ones(T, T, dtype=torch.uint8, device="cuda"))
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    fattn.fa_fwd_ex(g["q"], g["k"], g["v"], o2, lse2, None, opts, B, H, N, D, w.scale, True)
    g2 = [torch.empty_like(dq) for _ in range(3)]
    fattn.fa_bwd_ex(g["q"], g["k"], g["v"], o2, lse2, g["do"], *g2, None, opts, B, H, N, D,
                    w.scale, True, True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    for a, b in zip((dq, dk, dv), g2):
        assert torch.equal(a, b)


def test_block_mask_through_flash_attn_func():
    from exact_attention_93_gb300.attention import flash_attn_func
    B, H, N, D = 1, 2, 600, 64
    T = (N + 127) // 128
    mask = random_mask(T, 11, 0.5, keep_diagonal=True)
    w = W.custom(B, H, N, D, seed=25)
    inputs = W.make_inputs(w)
    q, k, v, do = (inputs[x].cuda().transpose(1, 2).contiguous() for x in ("q", "k", "v", "do"))
    for t in (q, k, v):
        t.requires_grad_()
    o = flash_attn_func(q, k, v, block_mask=torch.tensor(mask, device="cuda"))
    o.backward(do)
    torch.cuda.synchronize()
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], D ** -0.5, False,
                           dout=inputs["do"], block_mask=mask, block=128)
    assert U.o_err(o.detach().transpose(1, 2).float().cpu().numpy(), ref["o"], "bf16") <= U.TOL_O
    for t, name in ((q, "dq"), (k, "dk"), (v, "dv")):
        e = U.rel_err(t.grad.transpose(1, 2).float().cpu().numpy(), ref[name])
        assert e <= U.TOL_GRAD_REL, f"{name} {e:.3e}"
