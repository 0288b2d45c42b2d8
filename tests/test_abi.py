"""The C ABI on the host: libfattn.so builds, loads, exports every function
include/fattn.h declares, and rejects bad arguments before anything reaches
CUDA.  No kernel runs here."""
import ctypes
import subprocess

import pytest

from exact_attention_93_gb300 import build, fattn

NULL = None
EXPECTED = [
    "fa_abi_version", "fa_bwd", "fa_bwd_dkdv", "fa_bwd_dq", "fa_bwd_dq_convert", "fa_bwd_noalloc",
    "fa_bwd_ex", "fa_bwd_preprocess", "fa_bwd_strided", "fa_bwd_workspace_size", "fa_device_error",
    "fa_fwd", "fa_fwd_ex", "fa_fwd_fp8", "fa_fwd_fp8_workspace_size", "fa_fwd_strided",
    "fa_selftest_wait_timeout", "fa_status_string",
]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fattn.load()


def test_header_declares_the_expected_entry_points():
    assert fattn.declared_symbols() == sorted(EXPECTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fattn.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in fattn.declared_symbols():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_version_and_status_strings(lib):
    assert lib.fa_abi_version() == 5
    names = [lib.fa_status_string(i).decode() for i in range(5)]
    assert names == ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA",
                     "FA_ERR_TIMEOUT"]
    assert lib.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"


FAKE = 1 << 20  # an aligned, never dereferenced address: every case below fails before use


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, D=64, scale=0.125,
        causal=0, dtype=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, D, ctypes.c_float(scale), causal, dtype, NULL)


@pytest.mark.parametrize("kw,status", [
    ({"q": NULL}, fattn.FA_ERR_INVALID_ARG),
    ({"lse": NULL}, fattn.FA_ERR_INVALID_ARG),
    ({"v": FAKE + 8}, fattn.FA_ERR_INVALID_ARG),     # not 16-byte aligned
    ({"B": 0}, fattn.FA_ERR_INVALID_ARG),
    ({"H": -1}, fattn.FA_ERR_INVALID_ARG),
    ({"N": 0}, fattn.FA_ERR_INVALID_ARG),
    ({"D": 96}, fattn.FA_ERR_UNSUPPORTED),
    ({"D": 256}, fattn.FA_ERR_UNSUPPORTED),
    ({"dtype": 2}, fattn.FA_ERR_UNSUPPORTED),
    ({"scale": float("nan")}, fattn.FA_ERR_INVALID_ARG),
    ({"scale": float("inf")}, fattn.FA_ERR_INVALID_ARG),
    ({"B": 1 << 16, "H": 1 << 16}, fattn.FA_ERR_INVALID_ARG),   # B*H too large
    ({"B": 1 << 14, "H": 1 << 10, "N": 1 << 14, "D": 128}, fattn.FA_ERR_INVALID_ARG),
])
def test_fwd_rejects_bad_arguments(lib, kw, status):
    assert fwd(lib, **kw) == status


def test_workspace_size(lib):
    npad = 256
    base = 2 * ((3 * 4 * npad * 4 + 255) // 256 * 256)
    assert lib.fa_bwd_workspace_size(3, 4, 200, 64, 1) == base
    assert lib.fa_bwd_workspace_size(3, 4, 200, 64, 0) == base + (3 * 4 * 200 * 64 * 4 + 255) // 256 * 256
    assert lib.fa_bwd_workspace_size(3, 4, 200, 80, 0) == 0
    assert lib.fa_bwd_workspace_size(0, 4, 200, 64, 0) == 0


def bwd(lib, ws=FAKE, ws_bytes=1 << 40, D=64, deterministic=0, dq=FAKE, scale=0.125):
    return lib.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dq, FAKE, FAKE, 1, 1, 128, D,
                      ctypes.c_float(scale), 0, 0, deterministic, ws, ws_bytes, NULL)


def test_bwd_rejects_bad_arguments(lib):
    need = lib.fa_bwd_workspace_size(1, 1, 128, 64, 0)
    assert bwd(lib, ws=NULL) == fattn.FA_ERR_INVALID_ARG
    assert bwd(lib, ws=FAKE + 16) == fattn.FA_ERR_INVALID_ARG        # not 256-byte aligned
    assert bwd(lib, ws_bytes=need - 1) == fattn.FA_ERR_INVALID_ARG   # too small
    assert bwd(lib, dq=NULL) == fattn.FA_ERR_INVALID_ARG
    assert bwd(lib, D=32) == fattn.FA_ERR_UNSUPPORTED
    assert bwd(lib, scale=float("nan")) == fattn.FA_ERR_INVALID_ARG
    # the deterministic layout needs no dQ accumulator, so it is smaller
    det = lib.fa_bwd_workspace_size(1, 1, 128, 64, 1)
    assert det < need


def test_stage_entry_points_reject_bad_arguments(lib):
    f = ctypes.c_float(0.125)
    assert lib.fa_bwd_preprocess(NULL, FAKE, FAKE, 1, 1, 128, 64, 0, 0, FAKE, 1 << 40, NULL) == 1
    assert lib.fa_bwd_dkdv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, f, 0, 0, 0, FAKE, 10,
                           NULL) == 1
    assert lib.fa_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, f, 0, 0, NULL, 1 << 40,
                         NULL) == 1
    assert lib.fa_bwd_dq_convert(FAKE, 1, 1, 128, 64, f, 5, FAKE, 1 << 40, NULL) == 2
    code = ctypes.c_int(0)
    assert lib.fa_device_error(NULL, None) == 1
    assert lib.fa_selftest_wait_timeout(0, NULL) == 1
    assert lib.fa_selftest_wait_timeout(5000000, NULL) == 1
    del code


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fattn.fa_fwd(q, q, q, q, torch.zeros(1, 1, 128), 0.125, False)


def contiguous(B, H, N, D):
    return fattn.FaStrides(H * N * D, N * D, D)


def layout_with(**bad):
    c = contiguous(1, 2, 128, 64)
    L = fattn.FaLayout(*([c] * 8))
    for name, st in bad.items():
        setattr(L, name, st)
    return L


def fwd_strided(lib, L, B=1, H=2, N=128, D=64):
    return lib.fa_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, B, H, N, D, ctypes.byref(L),
                              ctypes.c_float(0.125), 0, 0, NULL)


def bwd_strided(lib, L, B=1, H=2, N=128, D=64):
    need = lib.fa_bwd_workspace_size(B, H, N, D, 0)
    return lib.fa_bwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, H, N, D,
                              ctypes.byref(L), ctypes.c_float(0.125), 0, 0, 0, FAKE, need, NULL)


@pytest.mark.parametrize("bad", [
    {"q": fattn.FaStrides(2 * 128 * 64, 128 * 64, 68)},    # seq stride not a multiple of 8
    {"k": fattn.FaStrides(2 * 128 * 64, 4, 64)},            # head stride not a multiple of 8
    {"v": fattn.FaStrides(-8, 128 * 64, 64)},               # negative
    {"o": fattn.FaStrides(0, 1 << 39, 64)},                # head 1 lies 2^40 bytes from the base
])
def test_strided_entry_points_reject_bad_strides(lib, bad):
    L = layout_with(**bad)
    assert fwd_strided(lib, L) == fattn.FA_ERR_INVALID_ARG
    assert bwd_strided(lib, L) == fattn.FA_ERR_INVALID_ARG


def test_strided_backward_checks_gradient_strides(lib):
    L = layout_with(dk=fattn.FaStrides(2 * 128 * 64, 128 * 64, 12))
    assert bwd_strided(lib, L) == fattn.FA_ERR_INVALID_ARG


def test_strided_entry_points_need_a_layout(lib):
    assert lib.fa_fwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, None,
                              ctypes.c_float(0.125), 0, 0, NULL) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_strided(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64,
                              None, ctypes.c_float(0.125), 0, 0, 0, FAKE, 1 << 40,
                              NULL) == fattn.FA_ERR_INVALID_ARG


def test_strides_of_reads_named_dimensions():
    torch = pytest.importorskip("torch")
    x = torch.zeros(2, 5, 3, 64)                      # (batch, seqlen, nheads, headdim)
    s = fattn.strides_of(x, "bnhd")
    assert (s.batch, s.head, s.seq) == (5 * 3 * 64, 64, 3 * 64)
    qkv = torch.zeros(2, 5, 3, 4, 128)                # packed (batch, seqlen, 3, nheads, headdim)
    k = qkv[:, :, 1]
    s = fattn.strides_of(k, "bnhd")
    assert (s.batch, s.head, s.seq) == (5 * 3 * 4 * 128, 128, 3 * 4 * 128)
    with pytest.raises(ValueError):
        fattn.strides_of(x.transpose(2, 3), "bnhd")   # D not contiguous


@pytest.mark.parametrize("win", [(-2, 0), (0, -2), (-5, -5)])
def test_ex_entry_points_reject_bad_windows(lib, win):
    opt = fattn.FaOptions(win[0], win[1], None, 0, None, 0)
    assert lib.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 128, 64, None, ctypes.byref(opt),
                         ctypes.c_float(0.125), 0, 0, NULL) == fattn.FA_ERR_INVALID_ARG
    need = lib.fa_bwd_workspace_size(1, 2, 128, 64, 0)
    assert lib.fa_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 128, 64, None,
                         ctypes.byref(opt), ctypes.c_float(0.125), 0, 0, 0, FAKE, need,
                         NULL) == fattn.FA_ERR_INVALID_ARG


def test_ex_entry_points_reject_misaligned_slopes(lib):
    opt = fattn.FaOptions(-1, -1, FAKE + 2, 0, None, 0)
    assert lib.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 128, 64, None, ctypes.byref(opt),
                         ctypes.c_float(0.125), 0, 0, NULL) == fattn.FA_ERR_INVALID_ARG


def test_block_mask_beyond_the_tile_limit_is_unsupported(lib):
    opt = fattn.FaOptions(-1, -1, None, 0, FAKE, 0)
    N = 128 * 16384 + 1                      # 16385 tiles along N
    assert lib.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, N, 64, None, ctypes.byref(opt),
                         ctypes.c_float(0.125), 0, 0, NULL) == fattn.FA_ERR_UNSUPPORTED


def fwd8(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=2, N=300, D=128, layout=None,
         opts=None, dq=None, dk=None, dv=None, scale=0.09, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.fa_fwd_fp8_workspace_size(B, H, N, 128)   # >= the D = 64 size
    return lib.fa_fwd_fp8(q, k, v, o, lse, B, H, N, D,
                          ctypes.byref(layout) if layout is not None else None,
                          ctypes.byref(opts) if opts is not None else None, dq, dk, dv,
                          ctypes.c_float(scale), 0, ws, ws_bytes, NULL)


def test_fp8_workspace_size(lib):
    # V^T: B*H*D*ld bytes, ld = N rounded up to 16, rounded up to 256
    assert lib.fa_fwd_fp8_workspace_size(1, 2, 300, 128) == 2 * 128 * 304
    assert lib.fa_fwd_fp8_workspace_size(3, 1, 1, 128) == 3 * 128 * 16
    assert lib.fa_fwd_fp8_workspace_size(1, 1, 130, 64) == 64 * 144
    assert lib.fa_fwd_fp8_workspace_size(1, 1, 128, 96) == 0     # D is 64 or 128
    assert lib.fa_fwd_fp8_workspace_size(0, 1, 128, 128) == 0


@pytest.mark.parametrize("kw,status", [
    ({"D": 96}, fattn.FA_ERR_UNSUPPORTED),
    ({"D": 32}, fattn.FA_ERR_UNSUPPORTED),
    ({"q": NULL}, fattn.FA_ERR_INVALID_ARG),
    ({"k": FAKE + 8}, fattn.FA_ERR_INVALID_ARG),
    ({"N": 0}, fattn.FA_ERR_INVALID_ARG),
    ({"scale": float("nan")}, fattn.FA_ERR_INVALID_ARG),
    ({"dv": FAKE + 2}, fattn.FA_ERR_INVALID_ARG),          # descale not 4-byte aligned
    ({"ws": NULL}, fattn.FA_ERR_INVALID_ARG),
    ({"ws": FAKE + 16}, fattn.FA_ERR_INVALID_ARG),          # workspace not 256-byte aligned
    ({"ws_bytes": 2 * 128 * 304 - 1}, fattn.FA_ERR_INVALID_ARG),
    # 8-bit operand strides are bytes and must be multiples of 16
    ({"layout": fattn.FaLayout(fattn.FaStrides(2 * 300 * 128, 300 * 128, 136),
                               *([fattn.FaStrides(2 * 300 * 128, 300 * 128, 128)] * 7))},
     fattn.FA_ERR_INVALID_ARG),
    ({"layout": fattn.FaLayout(*([fattn.FaStrides(2 * 300 * 128, 300 * 128, 128)] * 2),
                               fattn.FaStrides(2 * 300 * 128, 8, 128),
                               *([fattn.FaStrides(2 * 300 * 128, 300 * 128, 128)] * 5))},
     fattn.FA_ERR_INVALID_ARG),
    ({"opts": fattn.FaOptions(-3, 0, None, 0, None, 0)}, fattn.FA_ERR_INVALID_ARG),
])
def test_fp8_forward_rejects_bad_arguments(lib, kw, status):
    assert fwd8(lib, **kw) == status


def test_fp8_binding_checks_types():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fattn.fa_fwd_fp8(x, x, x, x, x, None, None, 1, 1, 128, 128, 0.1, False)  # CPU tensors
