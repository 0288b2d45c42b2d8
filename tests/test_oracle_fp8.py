"""Pins for the FP8 part of the oracle (``oracle.fp8``): the e4m3 decoder
against a library conversion and the format's landmark values, the
dequantisation factors against invariants of attention, the probability
rows against brute force; then planted mistakes in a copy of the module,
each of which some pin must catch.  CPU only."""
import importlib.util
import inspect
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8 as fp8
from exact_attention_93_gb300 import workloads as W


# --------------------------------------------------------------------------
# the decoder
# --------------------------------------------------------------------------

def pin_table_matches_torch(m=fp8):
    """Every byte decodes to what torch's float8_e4m3fn conversion gives."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = m.e4m3_decode(codes.numpy())
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # negative zero keeps its sign
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def pin_landmarks(m=fp8):
    """Values the format definition fixes (1 sign, 4 exponent bits with bias
    7, 3 mantissa bits, no infinities, S.1111.111 = NaN)."""
    v = m.e4m3_value
    assert v(0x38) == 1.0                      # 0.0111.000
    assert v(0x40) == 2.0
    assert v(0xC0) == -2.0
    assert v(0x3C) == 1.5                      # 0.0111.100
    assert v(0x7E) == 448.0                    # 0.1111.110, largest finite
    assert v(0x78) == 256.0                    # 0.1111.000
    assert v(0x08) == 2.0 ** -6                # smallest normal
    assert v(0x07) == 7 * 2.0 ** -9            # largest subnormal
    assert v(0x01) == 2.0 ** -9                # smallest subnormal
    assert v(0x00) == 0.0 and not math.copysign(1.0, v(0x00)) < 0
    assert v(0x80) == 0.0 and math.copysign(1.0, v(0x80)) < 0
    assert math.isnan(v(0x7F)) and math.isnan(v(0xFF))
    assert sum(math.isnan(v(c)) for c in range(256)) == 2


def pin_monotone(m=fp8):
    pos = np.array([m.e4m3_value(c) for c in range(0x00, 0x7F)])
    assert np.all(np.diff(pos) > 0)
    neg = np.array([m.e4m3_value(c) for c in range(0x80, 0xFF)])
    assert np.all(np.diff(neg) < 0)
    assert np.array_equal(neg, -pos)


def test_table_matches_torch():
    pin_table_matches_torch()


def test_landmarks():
    pin_landmarks()


def test_monotone_and_symmetric():
    pin_monotone()


def test_torch_float8_tensors_and_bytes_decode_alike():
    x = torch.randn(3, 5) * 40
    x8 = x.to(torch.float8_e4m3fn)
    assert np.array_equal(fp8.e4m3_decode(x8), fp8.e4m3_decode(x8.view(torch.uint8).numpy()))
    assert np.array_equal(fp8.e4m3_decode(x8), x8.to(torch.float64).numpy())


# --------------------------------------------------------------------------
# dequantisation and the attention it feeds
# --------------------------------------------------------------------------

def small_fp8(B=2, H=3, N=9, D=4, seed=3):
    w = W.custom(B, H, N, D, causal=False, seed=seed, backward=False)
    return W.make_fp8_inputs(w)


def brute_force(q, k, v, scale, causal):
    n = q.shape[0]
    s = scale * q @ k.T
    if causal:
        s = np.where(np.arange(n)[None, :] > np.arange(n)[:, None], -np.inf, s)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return p @ v, p


def pin_brute_force(m=fp8, causal=True):
    """O of the decoded, descaled inputs equals a direct numpy softmax."""
    d = small_fp8()
    res = m.attention_fp8(d["q8"], d["k8"], d["v8"], 0.3, causal, d["descale_q"], d["descale_k"],
                          d["descale_v"], want_probs=True)
    dq, dk, dv = (d[n].double().numpy() for n in ("descale_q", "descale_k", "descale_v"))
    for b in range(2):
        for h in range(3):
            q = d["q8"][b, h].to(torch.float64).numpy() * dq[b, h]
            k = d["k8"][b, h].to(torch.float64).numpy() * dk[b, h]
            v = d["v8"][b, h].to(torch.float64).numpy() * dv[b, h]
            o, p = brute_force(q, k, v, 0.3, causal)
            np.testing.assert_allclose(res["o"][b, h], o, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(res["p"][b, h], p, rtol=1e-12, atol=1e-15)


def pin_descale_invariants(m=fp8):
    """descale_v scales O; descale_q * descale_k acts as a factor on the
    scale; a factor of one head touches only that head."""
    d = small_fp8()
    fq, fk, fv = d["descale_q"], d["descale_k"], d["descale_v"]

    def run(scale, a=1.0, b=1.0, c=1.0):
        return m.attention_fp8(d["q8"], d["k8"], d["v8"], scale, False, fq * a, fk * b, fv * c)

    base = run(0.3)
    r = run(0.3, c=2.0)
    np.testing.assert_allclose(r["o"], 2.0 * base["o"], rtol=1e-13, atol=1e-300)
    np.testing.assert_array_equal(r["lse"], base["lse"])
    r = run(0.15, a=0.5, b=4.0)     # powers of two: the float32 factors stay exact
    ref = run(0.15 * 2.0)
    np.testing.assert_allclose(r["o"], ref["o"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["lse"], ref["lse"], rtol=1e-12)
    one = torch.ones(2, 3)
    one[1, 2] = 4.0
    r = run(0.3, c=one)
    mask = np.zeros((2, 3), bool)
    mask[1, 2] = True
    np.testing.assert_allclose(r["o"][mask], 4.0 * base["o"][mask], rtol=1e-13)
    np.testing.assert_array_equal(r["o"][~mask], base["o"][~mask])
    # a Q factor changes the weights, not the scale of O
    r = run(0.3, a=one)
    np.testing.assert_array_equal(r["o"][~mask], base["o"][~mask])
    assert np.max(np.abs(r["o"][mask] - base["o"][mask])) > 1e-3
    assert np.max(np.abs(r["o"][mask])) <= np.max(np.abs(
        m.dequantise(d["q8"], d["k8"], d["v8"], fq, fk, fv)[2][1, 2])) + 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force(causal):
    pin_brute_force(causal=causal)


def test_descale_invariants():
    pin_descale_invariants()


def test_probability_rows_match_the_outputs():
    rng = np.random.default_rng(11)
    q, k, v = (rng.standard_normal((40, 8)) for _ in range(3))
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 1, 1]], np.uint8)
    res = oracle.attention_head(q, k, v, 0.4, True, window=(9, -1), alibi_slope=0.1,
                                block_mask=bm, block=16, want_probs=True)
    p = res["p"]
    np.testing.assert_allclose(p @ v, res["o"], rtol=1e-12, atol=1e-13)
    sums = p.sum(axis=1)
    np.testing.assert_allclose(sums[sums > 0], 1.0, rtol=1e-13)
    i, j = np.meshgrid(np.arange(40), np.arange(40), indexing="ij")
    hidden = (j > i) | (j < i - 9) | (bm[i // 16, j // 16] == 0)
    assert np.all(p[hidden] == 0.0)
    # the probabilities are the exponentials of the scores minus the LSE
    s = 0.4 * q @ k.T - 0.1 * np.abs(i - j)
    fin = np.isfinite(res["lse"])
    vis = ~hidden & fin[:, None]
    np.testing.assert_allclose(p[vis], np.exp(s - res["lse"][:, None])[vis], rtol=1e-12)


def test_inputs_are_scaled_to_the_e4m3_range():
    d = small_fp8(B=1, H=2, N=300, D=128, seed=5)
    for n in ("q", "k", "v"):
        x = fp8.e4m3_decode(d[n + "8"])
        assert np.all(np.isfinite(x))
        assert np.max(np.abs(x)) == 448.0
        # the bytes times the factors reproduce the normal draws to e4m3 precision
        g = torch.Generator().manual_seed(5)
        draws = [torch.randn((1, 2, 300, 128), generator=g) for _ in range(3)]
        ref = draws["qkv".index(n)].double().numpy()
        deq = x * d["descale_" + n].double().numpy()[:, :, None, None]
        assert np.max(np.abs(deq - ref) / np.maximum(np.abs(ref), 1e-2)) < 2.0 ** -3


# --------------------------------------------------------------------------
# planted mistakes
# --------------------------------------------------------------------------

MUTANTS = [
    ("exponent bias 8", "2.0 ** (exponent - 7)", "2.0 ** (exponent - 8)"),
    ("subnormal scale 2^-7", "(mantissa / 8.0) * 2.0 ** -6", "(mantissa / 8.0) * 2.0 ** -7"),
    ("no implicit leading one", "(1.0 + mantissa / 8.0)", "(mantissa / 8.0)"),
    ("mantissa over 16", "(1.0 + mantissa / 8.0)", "(1.0 + mantissa / 16.0)"),
    ("sign ignored", "sign = -1.0 if code & 0x80 else 1.0", "sign = 1.0"),
    ("top exponent all NaN", "if exponent == 0xF and mantissa == 0x7:", "if exponent == 0xF:"),
    ("two mantissa bits", "mantissa = code & 0x7", "mantissa = code & 0x3"),
    ("exponent field misplaced", "exponent = (code >> 3) & 0xF", "exponent = (code >> 4) & 0x7"),
    ("Q and V factors swapped", "((q, descale_q), (k, descale_k), (v, descale_v))",
     "((q, descale_v), (k, descale_k), (v, descale_q))"),
    ("factors ignored", "out.append(x * _per_head(s, B, H)[:, :, None, None])", "out.append(x)"),
    ("factors by head only", "_per_head(s, B, H)[:, :, None, None]",
     "_per_head(s, B, H)[:1, :, None, None]"),
]

PINS = [pin_table_matches_torch, pin_landmarks, pin_monotone, pin_brute_force,
        pin_descale_invariants]


def load_variant(src):
    spec = importlib.util.spec_from_loader("oracle._fp8_variant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(src, os.path.join(os.path.dirname(fp8.__file__), "fp8_variant.py"), "exec"),
         mod.__dict__)
    return mod


def failing_pins(mod):
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except Exception:
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes_every_pin():
    assert failing_pins(load_variant(inspect.getsource(fp8))) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new):
    src = inspect.getsource(fp8)
    assert src.count(old) == 1, f"anchor for {name!r} not unique"
    assert failing_pins(load_variant(src.replace(old, new))), f"no pin caught {name!r}"
