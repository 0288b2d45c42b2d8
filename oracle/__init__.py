"""fp64 CPU reference for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares
no code with the CUDA library (``exact_attention_93_gb300``) and imports
nothing from it; the library never imports this.

The arithmetic lives in ``fa_oracle.c`` (plain C, double precision, OpenMP
over query rows).  This module compiles it with gcc on first use, or when
``build()`` is called, and marshals arrays through ctypes.

What is computed is the plain definition of attention (standard attention in
the l189.com "FlashAttention from scratch" walkthrough, sec. 1.1; causal mask
sec. 5.3; softmax Jacobian sec. 3.3), materialising the S and P rows of every
requested query row.  Pins against the pages and the mathematics are in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "libfa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into libfa_oracle.so next to it (gcc, -fopenmp)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)
            and os.path.getmtime(_LIB) >= os.path.getmtime(os.path.join(_HERE, "fa_oracle.h"))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    """ctypes handle with typed signatures for a compiled oracle at ``path``."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_long)
    lib.fa_oracle_rows.restype = ctypes.c_int
    lib.fa_oracle_rows.argtypes = [
        dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_double,
        ctypes.c_int, lp, ctypes.c_long, dp, dp, dp, dp, ctypes.c_long,
        ctypes.c_long, dp, dp,
    ]
    lib.fa_oracle_rows_ex.restype = ctypes.c_int
    lib.fa_oracle_rows_ex.argtypes = [
        dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_double,
        ctypes.c_int, ctypes.c_long, ctypes.c_long, ctypes.c_double, lp, ctypes.c_long,
        dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, dp, dp,
    ]
    lib.fa_oracle_rows_bs.restype = ctypes.c_int
    lib.fa_oracle_rows_bs.argtypes = [
        dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, ctypes.c_double,
        ctypes.c_int, ctypes.c_long, ctypes.c_long, ctypes.c_double,
        ctypes.POINTER(ctypes.c_ubyte), ctypes.c_long, lp, ctypes.c_long,
        dp, dp, dp, dp, ctypes.c_long, ctypes.c_long, dp, dp,
    ]
    lib.fa_oracle_rows_p.restype = ctypes.c_int
    lib.fa_oracle_rows_p.argtypes = list(lib.fa_oracle_rows_bs.argtypes) + [dp]
    lib.fa_oracle_threads.restype = ctypes.c_int
    lib.fa_oracle_threads.argtypes = []
    lib.fa_oracle_set_threads.restype = None
    lib.fa_oracle_set_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().fa_oracle_threads())


def set_threads(n: int) -> None:
    _load().fa_oracle_set_threads(int(n))


def _f64(a) -> np.ndarray:
    """Any array-like (numpy or torch, any float dtype) -> C-contiguous float64.

    bf16 and fp16 values are exactly representable in float64, so this upcast
    is exact."""
    if hasattr(a, "detach"):  # torch tensor, without importing torch here
        a = a.detach().to("cpu")
        if str(a.dtype) in ("torch.bfloat16", "torch.float16"):
            a = a.float()
        a = a.numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def attention_head(q, k, v, scale, causal, dout=None, rows=None,
                   kv_range=None, want_grads=True, window=(-1, -1), alibi_slope=0.0,
                   block_mask=None, block=128, want_probs=False):
    """Exact attention for one (batch, head) slice.

    q, k, v, dout: [N, D].  rows: query-row indices (default: all rows).
    kv_range: (begin, end) key range for dK/dV column sums (default: all keys
    when every row is requested, none otherwise).
    window: (left, right); query i sees keys i - left .. i + right, a
    negative bound being absent.  alibi_slope: the score of (i, j) gets
    -alibi_slope * |i - j| added after scaling.  block_mask: None or a
    [ceil(N / block), ceil(N / block)] array; key j is visible to query i
    only where block_mask[i // block, j // block] is nonzero.

    Returns a dict with o [R, D], lse [R], p [R, N] (the probability rows,
    when want_probs) and, when dout is given, dq [R, D], di [R] and (if a key
    range applies) dk, dv [end - begin, D].
    """
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 2 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [N, D] shape")
    N, D = q.shape
    do = _f64(dout) if dout is not None else None
    if do is not None and do.shape != q.shape:
        raise ValueError("dout must match q")
    if rows is None:
        rows_arr = None
        R = N
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).astype(np.int_)
        R = int(rows_arr.shape[0])
    o = np.empty((R, D), np.float64)
    lse = np.empty((R,), np.float64)
    dq = di = dk = dv = None
    kb = ke = 0
    if do is not None and want_grads:
        dq = np.empty((R, D), np.float64)
        di = np.empty((R,), np.float64)
        if kv_range is None and rows is None:
            kv_range = (0, N)
        if kv_range is not None:
            kb, ke = int(kv_range[0]), int(kv_range[1])
            dk = np.empty((ke - kb, D), np.float64)
            dv = np.empty((ke - kb, D), np.float64)
    left, right = (int(x) for x in window)
    bm = None
    if block_mask is not None:
        nb = (N + block - 1) // block
        bm = np.ascontiguousarray(np.asarray(block_mask) != 0, dtype=np.uint8)
        if bm.shape != (nb, nb):
            raise ValueError(f"block_mask must be [{nb}, {nb}] for N = {N}, block = {block}")
    probs = np.empty((R, N), np.float64) if want_probs else None
    rc = lib.fa_oracle_rows_p(
        _ptr(q), _ptr(k), _ptr(v), _ptr(do), N, D, float(scale), int(bool(causal)),
        left, right, float(alibi_slope),
        bm.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)) if bm is not None else None,
        int(block),
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long)) if rows_arr is not None else None,
        R, _ptr(o), _ptr(lse), _ptr(dq), _ptr(di), kb, ke, _ptr(dk), _ptr(dv), _ptr(probs))
    if rc != 0:
        raise RuntimeError(f"fa_oracle_rows_p failed with code {rc}")
    out = {"o": o, "lse": lse}
    if probs is not None:
        out["p"] = probs
    if dq is not None:
        out["dq"] = dq
        out["di"] = di
    if dk is not None:
        out["dk"] = dk
        out["dv"] = dv
    return out


def attention(q, k, v, scale, causal, dout=None, rows=None, kv_range=None,
              window=(-1, -1), alibi_slopes=None, block_mask=None, block=128,
              want_probs=False):
    """Exact attention over a [B, H, N, D] batch, one (b, h) slice at a time.

    rows: None (every row) or a callable (b, h) -> row indices, or an array of
    shape [B, H, R].  alibi_slopes: None, [H] or [B, H].  block_mask: None,
    [nb, nb] for every head, or [H, nb, nb].  Returns arrays shaped
    [B, H, R, ...]."""
    B, H, N, D = tuple(q.shape)
    slopes = np.zeros((B, H))
    if alibi_slopes is not None:
        a = _f64(alibi_slopes)
        slopes = np.broadcast_to(a, (B, H)) if a.ndim == 1 else a.reshape(B, H)
    res = {}
    for b in range(B):
        for h in range(H):
            if rows is None:
                r = None
            elif callable(rows):
                r = rows(b, h)
            else:
                r = rows[b][h]
            one = attention_head(q[b, h], k[b, h], v[b, h], scale, causal,
                                 None if dout is None else dout[b, h], r,
                                 kv_range, window=window, alibi_slope=slopes[b, h],
                                 block_mask=None if block_mask is None else
                                 (block_mask[h] if np.ndim(block_mask) == 3 else block_mask),
                                 block=block, want_probs=want_probs)
            for key, val in one.items():
                res.setdefault(key, []).append(val)
    for key in list(res):
        arrs = res[key]
        res[key] = np.stack(arrs).reshape((B, H) + arrs[0].shape)
    return res
