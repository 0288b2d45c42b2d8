"""flash_attn_func-style entry points with autograd.

The argument list follows the FlashAttention interface described by the
claire-chang.com introduction ([API]): q, k, v of shape
(batch, seqlen, nheads, headdim), softmax_scale defaulting to 1/sqrt(headdim),
causal, deterministic; and the packed variant taking one
(batch, seqlen, 3, nheads, headdim) tensor.  Both run the library's kernels
on the caller's tensors in place through the strided C ABI (fa_fwd_strided,
fa_bwd_ex): no transposes or copies of Q, K, V.  window_size gives
sliding-window local attention (query i sees keys i - left .. i + right,
-1 meaning no bound) and alibi_slopes ([nheads] or [batch, nheads] fp32) adds
-slope * |i - j| to each score, as the page documents.  block_mask (an
extension of that argument list) restricts attention to the kept blocks of
128 x 128 scores: block-sparse attention.  Dropout is not provided; asking
for it raises.  flash_attn_fp8_func is the forward on e4m3 inputs
(FlashAttention-3's FP8 forward, which the "Flash Attention" wiki page and
the v1 -> v3 table of "FlashAttention 深入" list), with per-(batch, head)
descale factors; it has no backward.
"""
from __future__ import annotations

import torch

from . import fattn

__all__ = ["flash_attn_func", "flash_attn_qkvpacked_func", "flash_attn_fp8_func"]


def _check_block_mask(block_mask, N, H):
    if block_mask is None:
        return None
    T = (N + 127) // 128
    if tuple(block_mask.shape) not in ((T, T), (H, T, T)):
        raise ValueError(f"block_mask must have shape ({T}, {T}) or ({H}, {T}, {T}) "
                         "for blocks of 128 x 128 scores")
    return block_mask.to(torch.uint8).contiguous()


def _check_options(dropout_p, window_size, alibi_slopes, B, H):
    if dropout_p:
        raise NotImplementedError("dropout is not supported (dropout_p must be 0)")
    left, right = (int(x) for x in window_size)
    if left < -1 or right < -1:
        raise ValueError("window_size bounds must be >= -1 (-1: no bound)")
    if alibi_slopes is not None:
        if tuple(alibi_slopes.shape) not in ((H,), (B, H)):
            raise ValueError("alibi_slopes must have shape (nheads,) or (batch, nheads)")
        alibi_slopes = alibi_slopes.to(torch.float32).contiguous()
    return (left, right), alibi_slopes


def _bnhd(t) -> fattn.FaStrides:
    return fattn.strides_of(t, "bnhd")


def _grad_operand(g):
    """The incoming gradient as the kernels need it: D contiguous, 16-byte
    aligned rows.  Anything else is copied once (argument marshalling)."""
    if g.stride(-1) != 1 or any(s % 8 for s in g.stride()[:-1]) or g.data_ptr() % 16:
        g = g.contiguous()
    return g


def _layout(q, k, v, o, do=None, dq=None, dk=None, dv=None) -> fattn.FaLayout:
    z = fattn.FaStrides(0, 0, 0)
    return fattn.FaLayout(_bnhd(q), _bnhd(k), _bnhd(v), _bnhd(o),
                          _bnhd(do) if do is not None else z, _bnhd(dq) if dq is not None else z,
                          _bnhd(dk) if dk is not None else z, _bnhd(dv) if dv is not None else z)


def _forward(q, k, v, scale, causal, window, slopes, bmask):
    B, N, H, D = (int(x) for x in q.shape)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same (batch, seqlen, nheads, headdim) shape")
    o = torch.empty((B, N, H, D), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fattn.fa_fwd_ex(q, k, v, o, lse, _layout(q, k, v, o), fattn.options(window, slopes, bmask),
                    B, H, N, D, scale, causal)
    return o, lse


def _backward(q, k, v, o, lse, do, dq, dk, dv, scale, causal, window, slopes, bmask,
              deterministic):
    B, N, H, D = (int(x) for x in q.shape)
    fattn.fa_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, _layout(q, k, v, o, do, dq, dk, dv),
                    fattn.options(window, slopes, bmask), B, H, N, D, scale, causal,
                    deterministic)


class _FlashAttn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, scale, causal, window, slopes, bmask, deterministic):
        o, lse = _forward(q, k, v, scale, causal, window, slopes, bmask)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.slopes, ctx.bmask = slopes, bmask
        ctx.scale, ctx.causal, ctx.window, ctx.deterministic = scale, causal, window, deterministic
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        _backward(q, k, v, o, lse, _grad_operand(do), dq, dk, dv, ctx.scale, ctx.causal,
                  ctx.window, ctx.slopes, ctx.bmask, ctx.deterministic)
        return dq, dk, dv, None, None, None, None, None, None


class _FlashAttnQKVPacked(torch.autograd.Function):
    @staticmethod
    def forward(ctx, qkv, scale, causal, window, slopes, bmask, deterministic):
        q, k, v = qkv.unbind(dim=2)
        o, lse = _forward(q, k, v, scale, causal, window, slopes, bmask)
        ctx.save_for_backward(qkv, o, lse)
        ctx.slopes, ctx.bmask = slopes, bmask
        ctx.scale, ctx.causal, ctx.window, ctx.deterministic = scale, causal, window, deterministic
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        qkv, o, lse = ctx.saved_tensors
        q, k, v = qkv.unbind(dim=2)
        dqkv = torch.empty_like(qkv)
        dq, dk, dv = dqkv.unbind(dim=2)
        _backward(q, k, v, o, lse, _grad_operand(do), dq, dk, dv, ctx.scale, ctx.causal,
                  ctx.window, ctx.slopes, ctx.bmask, ctx.deterministic)
        return dqkv, None, None, None, None, None, None


def flash_attn_func(q, k, v, dropout_p=0.0, softmax_scale=None, causal=False,
                    window_size=(-1, -1), alibi_slopes=None, deterministic=False,
                    return_lse=False, block_mask=None):
    """Exact attention of q, k, v shaped (batch, seqlen, nheads, headdim),
    bf16 or fp16 CUDA tensors with headdim 64 or 128 contiguous.  Returns the
    output in the same shape (and the fp32 (batch, nheads, seqlen) log-sum-exp
    of the scaled, biased scores when return_lse).  window_size = (left,
    right) limits query i to keys i - left .. i + right (-1: no bound);
    alibi_slopes adds -slope * |i - j|.  block_mask ((T, T) or (nheads, T, T),
    T = ceil(seqlen / 128)) keeps only the nonzero blocks of 128 x 128 scores.
    Differentiable in q, k, v (not in the slopes); deterministic selects the
    two-pass dQ backward."""
    window, slopes = _check_options(dropout_p, window_size, alibi_slopes, q.shape[0], q.shape[2])
    bmask = _check_block_mask(block_mask, q.shape[1], q.shape[2])
    scale = q.shape[-1] ** -0.5 if softmax_scale is None else float(softmax_scale)
    o, lse = _FlashAttn.apply(q, k, v, scale, bool(causal), window, slopes, bmask,
                              bool(deterministic))
    return (o, lse) if return_lse else o


def flash_attn_qkvpacked_func(qkv, dropout_p=0.0, softmax_scale=None, causal=False,
                              window_size=(-1, -1), alibi_slopes=None, deterministic=False,
                              return_lse=False, block_mask=None):
    """flash_attn_func on one packed (batch, seqlen, 3, nheads, headdim)
    tensor; its gradient comes back in the same packed layout."""
    if qkv.dim() != 5 or qkv.shape[2] != 3:
        raise ValueError("expected qkv of shape (batch, seqlen, 3, nheads, headdim)")
    window, slopes = _check_options(dropout_p, window_size, alibi_slopes, qkv.shape[0],
                                    qkv.shape[3])
    bmask = _check_block_mask(block_mask, qkv.shape[1], qkv.shape[3])
    scale = qkv.shape[-1] ** -0.5 if softmax_scale is None else float(softmax_scale)
    o, lse = _FlashAttnQKVPacked.apply(qkv, scale, bool(causal), window, slopes, bmask,
                                       bool(deterministic))
    return (o, lse) if return_lse else o


def flash_attn_fp8_func(q, k, v, softmax_scale=None, causal=False, window_size=(-1, -1),
                        alibi_slopes=None, block_mask=None, descale_q=None, descale_k=None,
                        descale_v=None, return_lse=False):
    """Forward-only attention of e4m3 q, k, v (torch.float8_e4m3fn, shaped
    (batch, seqlen, nheads, 64 or 128), head dim contiguous, other strides multiples
    of 16).  descale_q / descale_k / descale_v: None or fp32 (batch, nheads)
    factors; the result is attention of descale_q * q, descale_k * k and
    descale_v * v, returned in bf16 (with the fp32 (batch, nheads, seqlen)
    log-sum-exp when return_lse).  window_size, alibi_slopes and block_mask
    as for flash_attn_func."""
    B, N, H, D = (int(x) for x in q.shape)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must have the same (batch, seqlen, nheads, headdim) shape")
    window, slopes = _check_options(0.0, window_size, alibi_slopes, B, H)
    bmask = _check_block_mask(block_mask, N, H)
    desc = [None if t is None else t.to(torch.float32).reshape(B, H).contiguous()
            for t in (descale_q, descale_k, descale_v)]
    scale = D ** -0.5 if softmax_scale is None else float(softmax_scale)
    o = torch.empty((B, N, H, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    opts = fattn.options(window, slopes, bmask)
    fattn.fa_fwd_fp8(q, k, v, o, lse, _layout(q, k, v, o), opts, B, H, N, D, scale,
                     bool(causal), *desc)
    return (o, lse) if return_lse else o
