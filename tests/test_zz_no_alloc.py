"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (a plug-in inside another framework's step that gets only its tensors,
or a latency-bound caller that cannot afford cudaMalloc mid-step).  Its
scratch is a fixed array inside the library, shared by every call on a
device.

The GPU test compares two consecutive calls, on different shapes so that
the second call would see stale scratch contents if any leaked, with the
workspace-based deterministic fa_bwd on the same inputs.  This file is
collected last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import pytest
import torch

from exact_attention_93_gb300 import fattn, workloads as W
import parity_util as U

FAKE = 1 << 20  # aligned and never dereferenced: the call fails its checks first


def test_rejects_shapes_whose_scratch_does_not_fit():
    lib = fattn.load()
    # 17 heads x 65536 rows is past the 2^20 padded rows the scratch holds
    st = lib.fa_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 17, 65536,
                            128, ctypes.c_float(0.088), 1, fattn.FA_BF16, None)
    assert st == fattn.FA_ERR_UNSUPPORTED
    st = lib.fa_bwd_noalloc(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64,
                            ctypes.c_float(0.125), 0, fattn.FA_BF16, None)
    assert st == fattn.FA_ERR_INVALID_ARG


def _reference_and_noalloc(w):
    g = U.gpu_inputs(w, W.make_inputs(w))
    o, lse = U.run_forward(w, g)
    ref = U.run_backward(w, g, o, lse, True)  # workspace-based, deterministic
    got = tuple(torch.empty_like(g["q"]) for _ in range(3))
    fattn.fa_bwd_noalloc(g["q"], g["k"], g["v"], o, lse, g["do"], *got, w.scale, w.causal)
    torch.cuda.synchronize()
    return ref, got


@pytest.mark.gpu
def test_matches_workspace_backward_on_two_calls_in_a_row():
    shapes = [W.custom(2, 3, 1000, 128, dtype="bf16", causal=True, seed=21),
              W.custom(1, 2, 300, 64, dtype="fp16", causal=False, seed=22)]
    for w in shapes:
        ref, got = _reference_and_noalloc(w)
        for name, a, b in zip(("dq", "dk", "dv"), ref, got):
            r = a.float().cpu().numpy()
            err = U.rel_err(b.float().cpu().numpy(), r)
            assert err <= U.TOL_GRAD_REL, f"{w.name} {name}: {err:.3e}"
            # same kernels and order of summation as the deterministic path
            assert torch.equal(a, b), f"{w.name} {name} differs bitwise"
    assert fattn.fa_device_error() == fattn.FA_OK
