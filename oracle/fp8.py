"""fp64 reference for the FP8 forward -- TEST INFRASTRUCTURE ONLY.

Same rules as the rest of ``oracle``: only ``tests/``, ``smoke()`` and the
benchmark's CPU legs may import this, and it shares nothing with the CUDA
library.

What the FP8 forward computes (FlashAttention-3's FP8 forward, listed in the
implementation section of the "Flash Attention" wiki page and in the v3 row
of the v1 -> v3 table of "FlashAttention 深入"): attention of the
dequantised inputs,

    Q~ = descale_q[b, h] * value(Q),  K~ = descale_k[b, h] * value(K),
    V~ = descale_v[b, h] * value(V),  (O, LSE) = attention(Q~, K~, V~)

with the same masks, window, ALiBi bias and block mask as the 16-bit path.
The pages name no 8-bit format.  The reading taken is OCP FP8 E4M3 (the
"E4M3" format of Micikevicius et al., "FP8 Formats for Deep Learning", 2022,
which FlashAttention-3 takes): one sign bit, four exponent bits with bias 7,
three mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; the
all-ones pattern S.1111.111 is NaN and there are no infinities, so
S.1111.110 = 448 is the largest finite value.  ``e4m3_value`` writes that
definition out; the attention itself is the C oracle's.
"""
from __future__ import annotations

import numpy as np

from . import attention


def e4m3_value(code: int) -> float:
    """The real number one E4M3 byte encodes (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exponent = (code >> 3) & 0xF
    mantissa = code & 0x7
    if exponent == 0xF and mantissa == 0x7:
        return float("nan")
    if exponent == 0:
        return sign * (mantissa / 8.0) * 2.0 ** -6
    return sign * (1.0 + mantissa / 8.0) * 2.0 ** (exponent - 7)


# value of every byte, by code
E4M3 = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def as_bytes(a) -> np.ndarray:
    """E4M3 data (numpy uint8, or a torch float8_e4m3fn / uint8 tensor) as a
    numpy uint8 array of the same shape."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu")
        if a.dtype != torch.uint8:
            a = a.view(torch.uint8)
        a = a.numpy()
    a = np.asarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"expected e4m3 bytes, got {a.dtype}")
    return a


def e4m3_decode(a) -> np.ndarray:
    """float64 values of E4M3 data, elementwise."""
    return E4M3[as_bytes(a)]


def _per_head(x, B, H):
    if x is None:
        return np.ones((B, H))
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, np.float64).reshape(B, H)


def dequantise(q8, k8, v8, descale_q=None, descale_k=None, descale_v=None):
    """Q~, K~, V~ as float64 [B, H, N, D] from e4m3 [B, H, N, D] data and
    optional [B, H] factors (None: 1)."""
    q, k, v = e4m3_decode(q8), e4m3_decode(k8), e4m3_decode(v8)
    B, H = q.shape[:2]
    out = []
    for x, s in ((q, descale_q), (k, descale_k), (v, descale_v)):
        out.append(x * _per_head(s, B, H)[:, :, None, None])
    return tuple(out)


def attention_fp8(q8, k8, v8, scale, causal, descale_q=None, descale_k=None, descale_v=None,
                  **kw):
    """O and LSE (and whatever ``oracle.attention`` returns for ``kw``: rows,
    window, alibi_slopes, block_mask, want_probs) for e4m3 inputs."""
    q, k, v = dequantise(q8, k8, v8, descale_q, descale_k, descale_v)
    return attention(q, k, v, scale, causal, **kw)
