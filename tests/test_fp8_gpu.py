"""FP8 forward (fa_fwd_fp8) against the fp64 oracle on the dequantised
inputs, with the tolerance derived in ``fp8_bound``: every checked output
element inside the e4m3 bound, the root-mean-square error inside its
statistical allowance, LSE within 1e-3 plus the score allowance.  Inputs
are the seeded e4m3 draws of ``workloads.make_fp8_inputs``."""
import numpy as np
import pytest
import torch

import fp8_bound
import oracle
import oracle.fp8 as ofp8
from exact_attention_93_gb300 import attention, fattn, workloads as W

pytestmark = pytest.mark.gpu

D = 128


def run_fp8(d, B, H, N, scale, causal, opts=None, descale=True):
    q8, k8, v8 = (d[n].cuda() for n in ("q8", "k8", "v8"))
    D = q8.shape[-1]
    desc = [d["descale_" + n].cuda() if descale else None for n in "qkv"]
    o = torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    fattn.fa_fwd_fp8(q8, k8, v8, o, lse, None, opts, B, H, N, D, scale, causal, *desc)
    torch.cuda.synchronize()
    return o, lse


def check(d, o, lse, scale, causal, rows=None, descale=True, slopes=None, **kw):
    B, H, N = o.shape[:3]
    f = [d["descale_" + n] if descale else None for n in "qkv"]
    q, k, v = ofp8.dequantise(d["q8"], d["k8"], d["v8"], *f)
    o_np, lse_np = o.float().cpu().numpy(), lse.cpu().numpy()
    stats = []
    for b in range(B):
        for h in range(H):
            r = np.arange(N) if rows is None else np.asarray(rows[b][h])
            slope = 0.0 if slopes is None else float(slopes[h])
            ref = oracle.attention_head(q[b, h], k[b, h], v[b, h], scale, causal, rows=r,
                                        want_probs=True, alibi_slope=slope, **kw)
            stats.append(fp8_bound.check_head(o_np[b, h][r], lse_np[b, h][r], ref, q[b, h],
                                              k[b, h], v[b, h], scale, r, slope,
                                              label=f"b{b} h{h}"))
    ratio = max(s[0] for s in stats)
    print(f"max bound ratio {ratio:.3f}, rms {max(s[1] for s in stats):.2e} "
          f"(allowance {min(s[2] for s in stats):.2e})")
    return ratio


@pytest.mark.parametrize("B,H,N,D,causal,seed", [
    (1, 2, 300, 128, False, 21),
    (1, 2, 300, 128, True, 22),
    (2, 3, 1000, 128, True, 23),
    (1, 1, 1, 128, False, 24),
    (1, 2, 129, 128, True, 25),
    (2, 1, 128 * 5 + 17, 128, False, 26),
    (1, 2, 2048, 128, False, 27),
    (1, 2, 300, 64, False, 41),
    (2, 3, 1000, 64, True, 42),
    (1, 1, 1, 64, True, 43),
    (2, 1, 128 * 5 + 17, 64, False, 44),
    (1, 2, 2048, 64, True, 45),
])
def test_fp8_forward_within_the_e4m3_bound(B, H, N, D, causal, seed):
    d = W.make_fp8_inputs(W.custom(B, H, N, D, causal=causal, seed=seed, backward=False))
    scale = D ** -0.5
    o, lse = run_fp8(d, B, H, N, scale, causal)
    check(d, o, lse, scale, causal)


def test_fp8_head_dim_64_window_alibi_and_block_mask():
    B, H, N, D = 2, 2, 600, 64
    d = W.make_fp8_inputs(W.custom(B, H, N, D, causal=True, seed=46, backward=False))
    scale = D ** -0.5
    slopes = torch.tensor([0.5, 0.03125], dtype=torch.float32)
    opts = fattn.options((150, -1), slopes.cuda(), None)
    o, lse = run_fp8(d, B, H, N, scale, True, opts)
    check(d, o, lse, scale, True, slopes=slopes.numpy(), window=(150, -1))
    T = (N + 127) // 128
    mask = (np.random.default_rng(47).random((T, T)) < 0.6).astype(np.uint8)
    opts = fattn.options((-1, -1), None, torch.from_numpy(mask).cuda())
    o, lse = run_fp8(d, B, H, N, scale, False, opts)
    check(d, o, lse, scale, False, block_mask=mask)


def test_fp8_head_dim_64_api_layout_matches_contiguous_call_bit_for_bit():
    B, H, N, D = 2, 3, 333, 64
    d = W.make_fp8_inputs(W.custom(B, H, N, D, causal=False, seed=48, backward=False))
    o_ref, lse_ref = run_fp8(d, B, H, N, 0.11, False)
    q, k, v = (d[n + "8"].cuda().transpose(1, 2).contiguous() for n in "qkv")   # BNHD
    o, lse = attention.flash_attn_fp8_func(q, k, v, softmax_scale=0.11,
                                           descale_q=d["descale_q"].cuda(),
                                           descale_k=d["descale_k"].cuda(),
                                           descale_v=d["descale_v"].cuda(), return_lse=True)
    assert torch.equal(o.transpose(1, 2), o_ref)
    assert torch.equal(lse, lse_ref)


def test_fp8_forward_is_deterministic():
    d = W.make_fp8_inputs(W.custom(1, 2, 1000, D, causal=True, seed=31, backward=False))
    a = run_fp8(d, 1, 2, 1000, 0.1, True)
    b = run_fp8(d, 1, 2, 1000, 0.1, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_forward_without_descale_factors():
    """Bytes taken at face value (factors NULL), values of order one."""
    g = torch.Generator().manual_seed(32)
    B, H, N = 1, 2, 400
    d = {n + "8": (torch.randn(B, H, N, D, generator=g) * 0.7).to(torch.float8_e4m3fn)
         for n in "qkv"}
    o, lse = run_fp8(d, B, H, N, 0.09, False, descale=False)
    check(d, o, lse, 0.09, False, descale=False)


def test_fp8_forward_with_a_negative_scale():
    d = W.make_fp8_inputs(W.custom(1, 2, 333, D, causal=True, seed=33, backward=False))
    o, lse = run_fp8(d, 1, 2, 333, -0.05, True)
    check(d, o, lse, -0.05, True)


def test_fp8_window_alibi_and_block_mask():
    B, H, N = 1, 2, 700
    d = W.make_fp8_inputs(W.custom(B, H, N, D, causal=True, seed=34, backward=False))
    scale = D ** -0.5
    slopes = torch.tensor([0.25, 0.0625], dtype=torch.float32)
    opts = fattn.options((200, -1), slopes.cuda(), None)
    o, lse = run_fp8(d, B, H, N, scale, True, opts)
    check(d, o, lse, scale, True, slopes=slopes.numpy(), window=(200, -1))
    T = (N + 127) // 128
    rng = np.random.default_rng(35)
    mask = (rng.random((T, T)) < 0.5).astype(np.uint8)
    mask[2, :] = 0                      # a query block that sees nothing
    opts = fattn.options((-1, -1), None, torch.from_numpy(mask).cuda())
    o, lse = run_fp8(d, B, H, N, scale, False, opts)
    assert torch.all(o[:, :, 256:384] == 0)
    assert torch.all(torch.isneginf(lse[:, :, 256:384]))
    check(d, o, lse, scale, False, block_mask=mask)


def test_fp8_api_layout_matches_contiguous_call_bit_for_bit():
    """flash_attn_fp8_func on (batch, seqlen, nheads, headdim) views equals
    the contiguous [B, H, N, D] call exactly."""
    B, H, N = 2, 3, 500
    d = W.make_fp8_inputs(W.custom(B, H, N, D, causal=True, seed=36, backward=False))
    o_ref, lse_ref = run_fp8(d, B, H, N, 0.08, True)
    q, k, v = (d[n + "8"].cuda().transpose(1, 2).contiguous() for n in "qkv")   # BNHD
    o, lse = attention.flash_attn_fp8_func(q, k, v, softmax_scale=0.08, causal=True,
                                           descale_q=d["descale_q"].cuda(),
                                           descale_k=d["descale_k"].cuda(),
                                           descale_v=d["descale_v"].cuda(), return_lse=True)
    assert torch.equal(o.transpose(1, 2), o_ref)
    assert torch.equal(lse, lse_ref)


def test_fp8_full_size_sampled_rows():
    """The long-sequence causal shape (B1 H8 N65536 D128), in the launch
    configuration the benchmark times, checked on sampled rows."""
    w = W.WORKLOADS["long64k_causal"]
    d = W.make_fp8_inputs(w)
    o, lse = run_fp8(d, w.B, w.H, w.N, w.scale, True)
    rows = [[W.sampled_rows(w, b, h, count=62) for h in range(w.H)] for b in range(w.B)]
    check(d, o, lse, w.scale, True, rows=rows)
