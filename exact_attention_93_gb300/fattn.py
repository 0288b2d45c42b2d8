"""ctypes binding to libfattn.so (include/fattn.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  The functions take torch CUDA tensors (PyTorch
supplies device memory and streams) and pass raw pointers, sizes and the
current stream through the C ABI.  There is no fallback: if the library is
missing or cannot load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfattn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "fattn.h")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_BF16, FA_FP16 = 0, 1

_lock = threading.Lock()
_lib = None


class FaStrides(ctypes.Structure):
    """fa_strides: element strides (batch, head, seq) of one operand."""
    _fields_ = [("batch", ctypes.c_longlong), ("head", ctypes.c_longlong),
                ("seq", ctypes.c_longlong)]


class FaLayout(ctypes.Structure):
    """fa_layout: the strides of every operand of a call."""
    _fields_ = [(n, FaStrides) for n in ("q", "k", "v", "o", "dO", "dq", "dk", "dv")]


class FaOptions(ctypes.Structure):
    """fa_options: sliding window (-1 = no bound), ALiBi slopes, block mask."""
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("alibi_slopes", ctypes.c_void_p), ("alibi_per_batch", ctypes.c_int),
                ("block_mask", ctypes.c_void_p), ("block_mask_per_head", ctypes.c_int)]


class FattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = _status_name(status)
        super().__init__(f"{what} failed: {name} ({status})")


def _status_name(s: int) -> str:
    try:
        return load().fa_status_string(s).decode()
    except Exception:
        return str(s)


def declared_symbols() -> list[str]:
    """Every function include/fattn.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[a-z_ ]+\**\s*\**(fa_\w+)\(", text, re.M)))


def load(path: str | None = None):
    """Load libfattn.so (building it first if sources are newer) and set the
    argument types of every entry point."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if path is None:
            from . import build as _build
            if not _build.up_to_date():
                _build.build()
        if not os.path.exists(p):
            raise FileNotFoundError(f"libfattn.so not found at {p}; run build()")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "fa_abi_version": (i, []),
            "fa_status_string": (ctypes.c_char_p, [i]),
            "fa_fwd": (i, [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]),
            "fa_bwd_workspace_size": (sz, [i, i, i, i, i]),
            "fa_bwd": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp, sz, vp]),
            "fa_bwd_preprocess": (i, [vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]),
            "fa_bwd_dkdv": (i, [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp, sz, vp]),
            "fa_bwd_dq": (i, [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]),
            "fa_bwd_dq_convert": (i, [vp, i, i, i, i, f, i, vp, sz, vp]),
            "fa_device_error": (i, [vp, ctypes.POINTER(ctypes.c_int)]),
            "fa_selftest_wait_timeout": (i, [i, vp]),
            "fa_bwd_noalloc": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]),
            "fa_fwd_strided": (i, [vp, vp, vp, vp, vp, i, i, i, i, ctypes.POINTER(FaLayout), f,
                                   i, i, vp]),
            "fa_bwd_strided": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i,
                                   ctypes.POINTER(FaLayout), f, i, i, i, vp, sz, vp]),
            "fa_fwd_ex": (i, [vp, vp, vp, vp, vp, i, i, i, i, ctypes.POINTER(FaLayout),
                              ctypes.POINTER(FaOptions), f, i, i, vp]),
            "fa_bwd_ex": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i,
                              ctypes.POINTER(FaLayout), ctypes.POINTER(FaOptions), f, i, i, i,
                              vp, sz, vp]),
            "fa_fwd_fp8_workspace_size": (sz, [i, i, i, i]),
            "fa_fwd_fp8": (i, [vp, vp, vp, vp, vp, i, i, i, i, ctypes.POINTER(FaLayout),
                               ctypes.POINTER(FaOptions), vp, vp, vp, f, i, vp, sz, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


# --------------------------------------------------------------------------
# torch-facing helpers
# --------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float16")


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, D] tensors")
    return tuple(int(x) for x in q.shape)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str):
    if status != FA_OK:
        raise FattnError(status, what)


def _check_tensors(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libfattn takes CUDA tensors only")
        if not t.is_contiguous():
            raise ValueError("libfattn takes contiguous tensors only")


def strides_of(t, dims: str = "bhnd") -> FaStrides:
    """fa_strides of a 4-D tensor whose dimensions are named by `dims` (a
    permutation of "bhnd"); D must be the contiguous dimension."""
    if t.dim() != 4 or sorted(dims) != sorted("bhnd"):
        raise ValueError(f"expected a 4-D tensor and a permutation of 'bhnd', got {dims!r}")
    st = t.stride()
    if st[dims.index("d")] != 1:
        raise ValueError("the head dimension D must be contiguous")
    return FaStrides(st[dims.index("b")], st[dims.index("h")], st[dims.index("n")])


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libfattn takes CUDA tensors only")


def fa_fwd_strided(q, k, v, o, lse, layout: FaLayout, B: int, H: int, N: int, D: int,
                   scale: float, causal: bool, stream=None):
    """fa_fwd on operands in the layout `layout` (see fa_fwd_strided)."""
    _check_cuda(q, k, v, o, lse)
    st = load().fa_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D,
                               ctypes.byref(layout), float(scale), int(bool(causal)),
                               _dtype_code(q), _stream(stream))
    _check(st, "fa_fwd_strided")


def fa_bwd_strided(q, k, v, o, lse, do, dq, dk, dv, layout: FaLayout, B: int, H: int, N: int,
                   D: int, scale: float, causal: bool, deterministic: bool = False,
                   workspace=None, stream=None):
    """fa_bwd on operands in the layout `layout` (see fa_bwd_strided)."""
    _check_cuda(q, k, v, o, lse, do, dq, dk, dv, workspace)
    if workspace is None:
        workspace = alloc_workspace(B, H, N, D, deterministic, q.device)
    st = load().fa_bwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, D, ctypes.byref(layout),
                               float(scale), int(bool(causal)), _dtype_code(q),
                               int(bool(deterministic)), _ptr(workspace), workspace.numel(),
                               _stream(stream))
    _check(st, "fa_bwd_strided")


def options(window=(-1, -1), alibi_slopes=None, block_mask=None) -> FaOptions:
    """fa_options for a window (left, right), optional fp32 CUDA slopes of
    shape [H] or [B, H], and an optional uint8 CUDA block mask of shape
    [T, T] or [H, T, T], T = ceil(N / 128).  The returned object keeps the
    tensors it points at alive; the kernels read them when they run, so the
    caller keeps it (or the tensors) until the stream has passed the call."""
    opt = FaOptions(int(window[0]), int(window[1]), None, 0, None, 0)
    opt._tensors = (alibi_slopes, block_mask)
    if block_mask is not None:
        torch = _torch()
        if block_mask.dtype not in (torch.uint8, torch.bool) or not block_mask.is_cuda:
            raise ValueError("block_mask must be a uint8 or bool CUDA tensor")
        if not block_mask.is_contiguous() or block_mask.dim() not in (2, 3):
            raise ValueError("block_mask must be a contiguous [T, T] or [H, T, T] tensor")
        opt.block_mask = block_mask.data_ptr()
        opt.block_mask_per_head = 1 if block_mask.dim() == 3 else 0
    if alibi_slopes is not None:
        torch = _torch()
        if alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_cuda:
            raise ValueError("alibi_slopes must be a float32 CUDA tensor")
        if not alibi_slopes.is_contiguous() or alibi_slopes.dim() not in (1, 2):
            raise ValueError("alibi_slopes must be a contiguous [H] or [B, H] tensor")
        opt.alibi_slopes = alibi_slopes.data_ptr()
        opt.alibi_per_batch = 1 if alibi_slopes.dim() == 2 else 0
    return opt


def fa_fwd_ex(q, k, v, o, lse, layout, opts, B: int, H: int, N: int, D: int, scale: float,
              causal: bool, stream=None):
    """fa_fwd_ex: layout (FaLayout or None for contiguous) and options
    (FaOptions or None)."""
    _check_cuda(q, k, v, o, lse)
    st = load().fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D,
                          ctypes.byref(layout) if layout is not None else None,
                          ctypes.byref(opts) if opts is not None else None,
                          float(scale), int(bool(causal)), _dtype_code(q), _stream(stream))
    _check(st, "fa_fwd_ex")


def fa_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, layout, opts, B: int, H: int, N: int, D: int,
              scale: float, causal: bool, deterministic: bool = False, workspace=None,
              stream=None):
    """fa_bwd_ex, matching fa_fwd_ex."""
    _check_cuda(q, k, v, o, lse, do, dq, dk, dv, workspace)
    if workspace is None:
        workspace = alloc_workspace(B, H, N, D, deterministic, q.device)
    st = load().fa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                          _ptr(dk), _ptr(dv), B, H, N, D,
                          ctypes.byref(layout) if layout is not None else None,
                          ctypes.byref(opts) if opts is not None else None,
                          float(scale), int(bool(causal)), _dtype_code(q),
                          int(bool(deterministic)), _ptr(workspace), workspace.numel(),
                          _stream(stream))
    _check(st, "fa_bwd_ex")


def _check_fp8(*ts):
    torch = _torch()
    for t in ts:
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError(f"FP8 operands must be float8_e4m3fn (or their uint8 bytes), "
                            f"got {t.dtype}")


def _descale_ptr(t, B: int, H: int):
    if t is None:
        return None
    torch = _torch()
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.numel() != B * H:
        raise ValueError("descale factors must be contiguous float32 CUDA tensors of B*H "
                         "elements ([B, H])")
    return t.data_ptr()


def fa_fwd_fp8_workspace_size(B: int, H: int, N: int, D: int) -> int:
    return int(load().fa_fwd_fp8_workspace_size(B, H, N, D))


def alloc_fp8_workspace(B, H, N, D, device=None):
    """A 256-byte-aligned byte buffer of the size fa_fwd_fp8 needs."""
    torch = _torch()
    n = fa_fwd_fp8_workspace_size(B, H, N, D)
    if n == 0:
        raise ValueError("invalid sizes for an FP8 forward (D must be 64 or 128)")
    buf = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]


def fa_fwd_fp8(q, k, v, o, lse, layout, opts, B: int, H: int, N: int, D: int, scale: float,
               causal: bool, descale_q=None, descale_k=None, descale_v=None, workspace=None,
               stream=None):
    """fa_fwd_fp8: e4m3 q, k, v (float8_e4m3fn or uint8 bytes) in `layout`
    (FaLayout or None for contiguous [B, H, N, D]); o bf16; optional [B, H]
    float32 descale factors."""
    _check_cuda(q, k, v, o, lse, workspace)
    _check_fp8(q, k, v)
    if o.dtype != _torch().bfloat16:
        raise TypeError("the FP8 forward writes a bfloat16 O")
    dq_, dk_, dv_ = (_descale_ptr(t, B, H) for t in (descale_q, descale_k, descale_v))
    if workspace is None:
        workspace = alloc_fp8_workspace(B, H, N, D, q.device)
    st = load().fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D,
                           ctypes.byref(layout) if layout is not None else None,
                           ctypes.byref(opts) if opts is not None else None,
                           dq_, dk_, dv_, float(scale), int(bool(causal)), _ptr(workspace),
                           workspace.numel(), _stream(stream))
    _check(st, "fa_fwd_fp8")


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool, stream=None):
    """O and LSE for [B, H, N, D] q, k, v (see fa_fwd in include/fattn.h)."""
    _check_tensors(q, k, v, o, lse)
    B, H, N, D = _shape(q)
    st = load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D,
                       float(scale), int(bool(causal)), _dtype_code(q), _stream(stream))
    _check(st, "fa_fwd")


def fa_bwd_workspace_size(B: int, H: int, N: int, D: int, deterministic: bool) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, D, int(bool(deterministic))))


def alloc_workspace(B, H, N, D, deterministic, device=None):
    """A 256-byte-aligned byte buffer of the size fa_bwd needs (torch owns it)."""
    torch = _torch()
    n = fa_bwd_workspace_size(B, H, N, D, deterministic)
    if n == 0:
        raise ValueError("invalid sizes for a backward workspace")
    buf = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale: float, causal: bool,
           deterministic: bool = False, workspace=None, stream=None):
    """dQ, dK, dV (see fa_bwd in include/fattn.h)."""
    _check_tensors(q, k, v, o, lse, do, dq, dk, dv, workspace)
    B, H, N, D = _shape(q)
    if workspace is None:
        workspace = alloc_workspace(B, H, N, D, deterministic, q.device)
    st = load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                       _ptr(dk), _ptr(dv), B, H, N, D, float(scale), int(bool(causal)),
                       _dtype_code(q), int(bool(deterministic)), _ptr(workspace),
                       workspace.numel(), _stream(stream))
    _check(st, "fa_bwd")


def fa_bwd_preprocess(o, do, lse, deterministic, workspace, stream=None):
    B, H, N, D = _shape(o)
    st = load().fa_bwd_preprocess(_ptr(o), _ptr(do), _ptr(lse), B, H, N, D, _dtype_code(o),
                                  int(bool(deterministic)), _ptr(workspace), workspace.numel(),
                                  _stream(stream))
    _check(st, "fa_bwd_preprocess")


def fa_bwd_dkdv(q, k, v, do, dk, dv, scale, causal, deterministic, workspace, stream=None):
    B, H, N, D = _shape(q)
    st = load().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dk), _ptr(dv), B, H, N, D,
                            float(scale), int(bool(causal)), _dtype_code(q),
                            int(bool(deterministic)), _ptr(workspace), workspace.numel(),
                            _stream(stream))
    _check(st, "fa_bwd_dkdv")


def fa_bwd_dq(q, k, v, do, dq, scale, causal, workspace, stream=None):
    B, H, N, D = _shape(q)
    st = load().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), B, H, N, D,
                          float(scale), int(bool(causal)), _dtype_code(q), _ptr(workspace),
                          workspace.numel(), _stream(stream))
    _check(st, "fa_bwd_dq")


def fa_bwd_dq_convert(dq, scale, workspace, stream=None):
    B, H, N, D = _shape(dq)
    st = load().fa_bwd_dq_convert(_ptr(dq), B, H, N, D, float(scale), _dtype_code(dq),
                                  _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "fa_bwd_dq_convert")


def fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale: float, causal: bool, stream=None):
    """dQ, dK, dV with no workspace: for callers that cannot allocate device
    memory.  Same result as the deterministic fa_bwd; its scratch is a fixed
    array inside the library (see fa_bwd_noalloc in include/fattn.h for the
    size limit and the rule that overlapping calls race)."""
    _check_tensors(q, k, v, o, lse, do, dq, dk, dv)
    B, H, N, D = _shape(q)
    st = load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                               _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, D, float(scale),
                               int(bool(causal)), _dtype_code(q), _stream(stream))
    _check(st, "fa_bwd_noalloc")


def fa_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    code = ctypes.c_int(-1)
    st = load().fa_device_error(_stream(stream), ctypes.byref(code))
    _check(st, "fa_device_error")
    return code.value


def fa_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    """Run the bounded-wait self test; returns its status (FA_ERR_TIMEOUT when
    the wait ran out as designed)."""
    return int(load().fa_selftest_wait_timeout(int(limit_us), _stream(stream)))


# --------------------------------------------------------------------------
# Convenience wrappers that allocate outputs (torch owns the memory)
# --------------------------------------------------------------------------

def forward(q, k, v, scale=None, causal=False, stream=None):
    """Returns (o, lse).  scale defaults to 1/sqrt(D)."""
    torch = _torch()
    B, H, N, D = _shape(q)
    if scale is None:
        scale = D ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, scale, causal, stream)
    return o, lse


def backward(q, k, v, o, lse, do, scale=None, causal=False, deterministic=False, stream=None):
    """Returns (dq, dk, dv)."""
    torch = _torch()
    D = q.shape[-1]
    if scale is None:
        scale = D ** -0.5
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd(q, k, v, o, lse, do, dq, dk, dv, scale, causal, deterministic, stream=stream)
    return dq, dk, dv
