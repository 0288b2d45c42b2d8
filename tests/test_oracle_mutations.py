"""Plant plausible mistakes in a copy of the oracle's C source and check that
the pins catch every one.  Each mutant is compiled on the CPU into a temporary
directory; the real oracle is untouched."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "fa_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("causal mask includes no diagonal", "if (causal && j > i)", "if (causal && j >= i)"),
    ("causal mask off", "if (causal && j > i)", "if (causal && j > i + 1000000000L)"),
    ("scale dropped from scores", "s_row[j] = scale * acc", "s_row[j] = acc"),
    ("no max shift", "if (s_row[j] > m) m = s_row[j];", "if (s_row[j] > m) m = 0.0;"),
    ("softmax not normalised", "for (long j = 0; j < N; ++j) p_row[j] /= denom;", ";"),
    ("lse misses the max", "? m + log(denom)", "? log(denom)"),
    ("output uses keys instead of values", "const double* vj = v + j * D;\n        for (long d = 0; d < D; ++d) o_i[d]",
     "const double* vj = k + j * D;\n        for (long d = 0; d < D; ++d) o_i[d]"),
    ("dP uses keys", "for (long d = 0; d < D; ++d) acc += doi[d] * vj[d];",
     "for (long d = 0; d < D; ++d) acc += doi[d] * (k + j * D)[d];"),
    ("dS drops Di", "ds_row[j] = p_row[j] * (ds_row[j] - di);", "ds_row[j] = p_row[j] * ds_row[j];"),
    ("dS wrong sign", "ds_row[j] = p_row[j] * (ds_row[j] - di);", "ds_row[j] = p_row[j] * (di - ds_row[j]);"),
    ("Di block-local partial sum", "for (long j = 0; j < N; ++j) di += p_row[j] * ds_row[j];",
     "for (long j = 0; j < (N + 1) / 2; ++j) di += p_row[j] * ds_row[j];"),
    ("dQ uses values", "const double* kj = k + j * D;\n            for (long d = 0; d < D; ++d) dq_i[d]",
     "const double* kj = v + j * D;\n            for (long d = 0; d < D; ++d) dq_i[d]"),
    ("dQ misses scale", "for (long d = 0; d < D; ++d) dq_i[d] *= scale;", ";"),
    ("dK misses scale", "for (long d = 0; d < D; ++d) dkj[d] *= scale;", ";"),
    ("dV uses dS", "double p = p_all[(size_t)r * N + j];", "double p = ds_all[(size_t)r * N + j];"),
    ("dK uses dO", "const double* qi = q + i * D;\n                    for", "const double* qi = dout + i * D;\n                    for"),
    ("window left bound off by one", "j < i - left", "j <= i - left"),
    ("window left bound ignored", "if (left >= 0 && j < i - left) return 0;", ";"),
    ("window right bound ignored", "if (right >= 0 && j > i + right) return 0;", ";"),
    ("window bounds swapped", "j > i + right", "j > i + left"),
    ("alibi sign flipped", "- slope * (double)labs(i - j)", "+ slope * (double)labs(i - j)"),
    ("alibi without absolute value", "(double)labs(i - j)", "(double)(i - j)"),
    ("alibi scaled with the scores", "s_row[j] = scale * acc - slope * (double)labs(i - j);",
     "s_row[j] = scale * (acc - slope * (double)labs(i - j));"),
    ("block mask ignored", "if (bm->mask && !bm->mask[(i / bm->tile) * bm->n_kb + j / bm->tile]) return 0;", ";"),
    ("block mask transposed", "bm->mask[(i / bm->tile) * bm->n_kb + j / bm->tile]",
     "bm->mask[(j / bm->tile) * bm->n_kb + i / bm->tile]"),
    ("empty row divides by zero", "if (denom > 0.0)\n        for", "if (1)\n        for"),
]


def run_pins():
    """A battery of pins; returns the names of the ones that fail."""
    failed = []
    checks = [
        ("brute_force", lambda: pins.test_brute_force_tiny(5, 2, True)),
        ("brute_force_nc", lambda: pins.test_brute_force_tiny(7, 4, False)),
        ("row_sums", lambda: pins.test_probability_rows_sum_to_one_and_respect_mask(True)),
        ("zero_scale", lambda: pins.test_zero_scale_is_mean_of_visible_values(True)),
        ("large_scores", pins.test_large_scores_concentrate_on_the_argmax_without_overflow),
        ("sdpa_c", lambda: pins.test_matches_torch_sdpa_float64_forward_and_gradients(19, 8, True)),
        ("sdpa_nc", lambda: pins.test_matches_torch_sdpa_float64_forward_and_gradients(19, 8, False)),
        ("finite_diff", lambda: pins.test_gradients_by_central_differences(4, 3, True)),
        ("invariants", lambda: pins.test_gradient_invariants_and_di_identity(True)),
        ("band_bf", lambda: pins.test_window_and_alibi_brute_force(2, 1, 0.0, False)),
        ("band_bf_c", lambda: pins.test_window_and_alibi_brute_force(3, -1, 0.0, True)),
        ("alibi_bf", lambda: pins.test_window_and_alibi_brute_force(2, 3, 0.25, False)),
        ("band_sdpa", lambda: pins.test_window_and_alibi_match_torch_sdpa_float64(5, 3, 0.0, False)),
        ("alibi_closed", pins.test_alibi_at_zero_scale_is_a_closed_form),
        ("blocks_bf", lambda: pins.test_block_mask_brute_force(9, 3, 2, False)),
        ("blocks_sdpa", lambda: pins.test_block_mask_matches_torch_sdpa_float64(True)),
        ("blocks_empty", pins.test_rows_that_see_no_key_are_zero_and_carry_no_gradient),
    ]
    for name, fn in checks:
        try:
            with np.errstate(all="ignore"):
                fn()
        except Exception:  # an assertion, or NaNs tripping one
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_the_battery():
    assert run_pins() == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path, monkeypatch):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    mutated = src.replace(old, new, 1)
    assert mutated != src
    shutil.copy(os.path.join(os.path.dirname(SRC), "fa_oracle.h"), tmp_path / "fa_oracle.h")
    (tmp_path / "fa_oracle.c").write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-o", str(so),
                    str(tmp_path / "fa_oracle.c"), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle._bind(str(so)))
    failed = run_pins()
    assert failed, f"no pin caught the planted mistake: {name}"
