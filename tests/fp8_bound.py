"""Tolerance of the FP8 forward, derived from its arithmetic.

The pages give no tolerance for FP8 inputs, so the bound is derived here
from what the kernel computes, against the oracle's exact attention of the
dequantised inputs Q~, K~, V~ (``oracle.fp8``).

The kernel forms every score from exact e4m3 products accumulated in fp32,
keeps the softmax statistics in fp32, and enters the probabilities into the
P V product rounded to e4m3: P_j = 2^(x_j - m + 4) in log2 units, with the
reference maximum m at most 4 below the running maximum, so P < 256 (no
saturation at 448) and a weight stays normal (>= 2^-6) down to 2^-10 of the
running maximum.  The row sum l uses the unrounded P.

Per output element (i, d), with w_j the exact softmax weights of row i:

  (a) P rounding.  e4m3 has 3 mantissa bits: half an ulp is at most 2^-4 of
      the value in the normal range; the subnormal spacing is 2^-9, so a P
      below 2^-6 moves by at most min(P, 2^-10).  The final row sum is at
      least 2^4 / w_max (the largest weight's P is >= 2^4 after the last
      rescale), so in normalised units key j moves by at most
          eps_j = max(2^-4 w_j, min(w_j, 2^-14 w_max))
      and O by at most  sum_j eps_j |V~_jd|.
  (b) Scores.  An allowance of 2^-12 of sum_d |Q~_id K~_jd| * |scale| for the
      fp32 accumulation of D products (round-off of a plain fp32 sum is below
      2^-17 of it), plus 2^-22 of |x_ij| for forming the biased score in
      fp32.  If every score of row i moves by at most delta_i, every weight
      moves by a factor within exp(+-2 delta_i):  (e^(2 delta_i) - 1) *
      sum_j w_j |V~_jd|.
  (c) The fp32 accumulation of P V over the keys: an allowance of 2^-12 of
      sum_j w_j |V~_jd|.
  (d) O is rounded to bf16: half an ulp, at most 2^-8 of |O_d| plus the
      above.

Statistical check.  If the rounding errors in (a) are independent with mean
zero (round to nearest of values that are not on the grid), the error of
element (i, d) from (a) has variance at most sigma^2 = sum_j eps_j^2
|V~_jd|^2.  Over many elements the root-mean-square error must then stay
below twice sqrt(mean sigma^2) plus the root-mean-square of (b) + (c) + (d).
A bias in the rounding (every P rounded down, a wrong scale of P) breaks
this long before it breaks the elementwise bound.

LSE carries no P rounding: |LSE - LSE_ref| <= 1e-3 (the 16-bit bound) +
delta_i.
"""
import numpy as np

E4M3_REL = 2.0 ** -4        # half an ulp of e4m3, relative, normal range
E4M3_SUB_REL = 2.0 ** -14   # 2^-10 absolute in P units over a row sum >= 2^4 / w_max
GAMMA_S = 2.0 ** -12        # fp32 accumulation allowance for a score
GAMMA_X = 2.0 ** -22        # forming the biased score in fp32
GAMMA_PV = 2.0 ** -12       # fp32 accumulation allowance for P V
BF16_HALF_ULP = 2.0 ** -8   # relative
TOL_LSE = 1e-3


def score_delta(q, k, scale, rows, slope=0.0):
    """delta_i of (b) for query rows ``rows`` of one head (q, k: [N, D]
    dequantised)."""
    aq, ak = np.abs(q[rows]), np.abs(k)
    mag = abs(scale) * (aq @ ak.T)                                    # [R, N]
    far = np.abs(np.asarray(rows)[:, None] - np.arange(k.shape[0])[None, :])
    xmax = np.max(mag + abs(slope) * far, axis=1)
    return GAMMA_S * np.max(mag, axis=1) + GAMMA_X * xmax


def o_bound(p, v, o_ref, delta):
    """Elementwise bound on |O - O_ref| and the statistical sigma^2 of (a).

    p: [R, N] exact weights (oracle), v: [N, D] dequantised values,
    o_ref: [R, D], delta: [R].  Returns (bound [R, D], sigma2 [R, D],
    deterministic part [R, D])."""
    wmax = np.max(p, axis=1, keepdims=True)
    eps = np.maximum(E4M3_REL * p, np.minimum(p, E4M3_SUB_REL * wmax))   # [R, N]
    av = np.abs(v)
    a = eps @ av
    wv = p @ av
    det = (np.expm1(2.0 * delta)[:, None] + GAMMA_PV) * wv
    bound = a + det
    bound = bound + BF16_HALF_ULP * (np.abs(o_ref) + bound) + 1e-7
    sigma2 = (eps * eps) @ (av * av)
    return bound, sigma2, det + BF16_HALF_ULP * np.abs(o_ref)


def check_head(o, lse, ref, q, k, v, scale, rows, slope=0.0, label=""):
    """Assert the FP8 result of one head (o [R, D], lse [R], numpy) against
    the oracle's ``ref`` (o, lse, p for the same rows).  Returns
    (max bound ratio, rms error, rms allowance)."""
    rows = np.asarray(rows)
    delta = score_delta(q, k, scale, rows, slope)
    bound, sigma2, det = o_bound(ref["p"], v, ref["o"], delta)
    err = np.abs(np.asarray(o, np.float64) - ref["o"])
    ratio = float(np.max(err / bound))
    assert ratio <= 1.0, f"{label}: O outside the e4m3 bound (max ratio {ratio:.3f})"
    rms = float(np.sqrt(np.mean(err * err)))
    allow = 2.0 * float(np.sqrt(np.mean(sigma2))) + float(np.sqrt(np.mean(det * det)))
    assert rms <= allow, f"{label}: rms error {rms:.3e} above {allow:.3e}"
    lref = ref["lse"]
    lse = np.asarray(lse, np.float64)
    finite = np.isfinite(lref)
    assert np.array_equal(np.isfinite(lse), finite), f"{label}: LSE finiteness differs"
    lerr = np.abs(lse[finite] - lref[finite])
    assert np.all(lerr <= TOL_LSE + delta[finite]), f"{label}: LSE error {lerr.max():.3e}"
    return ratio, rms, allow
