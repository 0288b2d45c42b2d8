"""Pins for the fp64 oracle: values the pages print, closed forms, special
cases, brute force, a library routine, an independent blockwise online-softmax
recomputation and finite differences.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------------------
# The worked online-softmax example (l189.com walkthrough, sec. 2.2)
# --------------------------------------------------------------------------

def blockwise_softmax_trace(x, bs):
    """Online softmax over a score row, block by block, as the page's prose
    describes it: keep the running maximum m and the running sum l; when a
    block raises the maximum, scale the old sum by exp(m_old - m_new)."""
    trace = []
    m, l = -math.inf, 0.0
    for s in range(0, len(x), bs):
        blk = x[s:s + bs]
        m_new = max(m, max(blk))
        corr = 0.0 if m == -math.inf else l * math.exp(m - m_new)
        e = [math.exp(t - m_new) for t in blk]
        trace.append({"m": m_new, "e": e, "l_block": sum(e), "l_old_corrected": corr,
                      "local": [t / sum(e) for t in e]})
        l = corr + sum(e)
        m = m_new
    final = [math.exp(t - m) / l for t in x]
    return trace, l, final


def oracle_softmax_row(x):
    """softmax of one score row through the oracle: Q_0 = e_0, K_j = x_j e_0,
    V = identity, scale 1, so O_0 = P_0 and LSE_0 = logsumexp(x)."""
    n = len(x)
    q = np.zeros((n, n))
    q[0, 0] = 1.0
    k = np.zeros((n, n))
    k[:, 0] = x
    v = np.eye(n)
    r = oracle.attention_head(q, k, v, 1.0, False, rows=[0])
    return r["o"][0], r["lse"][0]


def test_worked_example_intermediates_match_page():
    g = json.load(open(os.path.join(GOLDEN, "online_softmax_worked_example.json")))
    pr, tol = g["printed"], g["print_tolerance"]
    trace, l_total, final = blockwise_softmax_trace(g["scores"], g["block_size"])
    b1, b2 = trace
    assert b1["m"] == pytest.approx(pr["m1"], abs=tol)
    assert b1["e"] == pytest.approx(pr["e1"], abs=tol)
    assert b1["l_block"] == pytest.approx(pr["l1"], abs=tol)
    assert b1["local"] == pytest.approx(pr["local_softmax_block1"], abs=tol)
    assert b2["m"] == pytest.approx(pr["m2_new"], abs=tol)
    assert b2["l_old_corrected"] == pytest.approx(pr["l1_corrected"], abs=tol)
    assert b2["l_block"] == pytest.approx(pr["l2"], abs=tol)
    assert l_total == pytest.approx(pr["l_total"], abs=tol)


def test_worked_example_oracle_is_softmax_and_agrees_with_page_where_page_is_right():
    g = json.load(open(os.path.join(GOLDEN, "online_softmax_worked_example.json")))
    x, pr, tol = g["scores"], g["printed"], g["print_tolerance"]
    p, lse = oracle_softmax_row(x)
    ex = np.exp(np.array(x) - 5.0)
    truth = ex / ex.sum()
    # the exact softmax, computed here independently
    np.testing.assert_allclose(p, truth, rtol=0, atol=1e-15)
    assert lse == pytest.approx(5.0 + math.log(ex.sum()), abs=1e-14)
    # the online recomputation reaches the same vector
    _, _, final = blockwise_softmax_trace(x, g["block_size"])
    np.testing.assert_allclose(p, final, rtol=0, atol=1e-15)
    # where the printed vector is right: the third entry, and block 1's share
    assert p[2] == pytest.approx(pr["final"][2], abs=tol)
    assert p[0] + p[1] == pytest.approx(pr["final"][0], abs=tol)
    # where it is not: entries 0, 1, 3 as printed are not the softmax, and the
    # printed vector's ratios contradict exp(2-1) = p0/p1 and exp(3-2) = p3/p0.
    for idx in (0, 1, 3):
        assert abs(p[idx] - pr["final"][idx]) > 10 * tol
    assert p[0] / p[1] == pytest.approx(math.e, rel=1e-12)
    assert p[3] / p[0] == pytest.approx(math.e, rel=1e-12)


# --------------------------------------------------------------------------
# Brute force, written independently with math.exp on tiny inputs
# --------------------------------------------------------------------------

def brute_force(q, k, v, scale, causal):
    n, d = q.shape
    o = np.zeros((n, d))
    lse = np.zeros(n)
    for i in range(n):
        s = []
        for j in range(n):
            if causal and j > i:
                continue
            s.append((j, scale * sum(q[i, t] * k[j, t] for t in range(d))))
        z = sum(math.exp(val) for _, val in s)
        lse[i] = math.log(z)
        for j, val in s:
            for t in range(d):
                o[i, t] += math.exp(val) / z * v[j, t]
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 1), (2, 3), (5, 2), (7, 4)])
def test_brute_force_tiny(n, d, causal):
    q, k, v = rnd((n, d), 1), rnd((n, d), 2), rnd((n, d), 3)
    scale = 0.7
    o_bf, lse_bf = brute_force(q, k, v, scale, causal)
    r = oracle.attention_head(q, k, v, scale, causal)
    np.testing.assert_allclose(r["o"], o_bf, rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["lse"], lse_bf, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# Rows of P sum to one (V = identity exposes P as O)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one_and_respect_mask(causal):
    n = 24
    q, k = rnd((n, n), 4, 2.0), rnd((n, n), 5, 2.0)
    r = oracle.attention_head(q, k, np.eye(n), 0.5, causal)
    p = r["o"]
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    if causal:
        assert np.all(np.triu(p, 1) == 0.0)
        assert np.all(np.diag(p) > 0)


# --------------------------------------------------------------------------
# Independent blockwise online-softmax attention (the exactness claim)
# --------------------------------------------------------------------------

def online_attention(q, k, v, scale, causal, bs):
    """Tiled attention with a running max / running sum per row, starting from
    m = -inf, l = 0 so that the first block reduces to a plain softmax."""
    n, d = q.shape
    o = np.zeros((n, d))
    lse = np.zeros(n)
    for i in range(n):
        m, l, acc = -math.inf, 0.0, np.zeros(d)
        for s in range(0, n, bs):
            e = min(s + bs, n)
            sc = scale * (k[s:e] @ q[i])
            if causal:
                sc = np.where(np.arange(s, e) <= i, sc, -np.inf)
            if np.all(sc == -np.inf):
                continue
            m_new = max(m, sc.max())
            alpha = 0.0 if m == -math.inf else math.exp(m - m_new)
            p = np.exp(sc - m_new)
            l = alpha * l + p.sum()
            acc = alpha * acc + p @ v[s:e]
            m = m_new
        o[i] = acc / l
        lse[i] = m + math.log(l)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bs", [1, 2, 3, 64, 70])
def test_online_recomputation_matches_full_softmax(bs, causal):
    n, d = 70, 8
    q, k, v = rnd((n, d), 6, 1.5), rnd((n, d), 7, 1.5), rnd((n, d), 8)
    r = oracle.attention_head(q, k, v, 0.9, causal)
    o_on, lse_on = online_attention(q, k, v, 0.9, causal, bs)
    np.testing.assert_allclose(r["o"], o_on, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["lse"], lse_on, rtol=0, atol=1e-12)


def test_minus_inf_initialisation_makes_first_block_a_plain_softmax():
    """(l189.com walkthrough, sec. 3.1) with m = -inf and l = 0 the first merge
    has correction factor exp(-inf) = 0, so one block of keys gives softmax."""
    n, d = 6, 3
    q, k, v = rnd((n, d), 9), rnd((n, d), 10), rnd((n, d), 11)
    o1, lse1 = online_attention(q, k, v, 1.0, False, n)  # a single block
    assert math.exp(-math.inf) == 0.0
    r = oracle.attention_head(q, k, v, 1.0, False)
    np.testing.assert_allclose(r["o"], o1, rtol=0, atol=1e-14)
    np.testing.assert_allclose(r["lse"], lse1, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# Closed forms and special cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_give_constant_output(causal):
    n, d = 33, 5
    c = rnd((d,), 12)
    r = oracle.attention_head(rnd((n, d), 13), rnd((n, d), 14), np.tile(c, (n, 1)), 0.3, causal)
    np.testing.assert_allclose(r["o"], np.tile(c, (n, 1)), rtol=0, atol=1e-13)


def test_single_key_gives_value_and_its_score():
    q, k, v = rnd((1, 7), 15), rnd((1, 7), 16), rnd((1, 7), 17)
    r = oracle.attention_head(q, k, v, 0.25, False)
    np.testing.assert_allclose(r["o"], v, rtol=0, atol=0)
    assert r["lse"][0] == pytest.approx(0.25 * float(q[0] @ k[0]), abs=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_mean_of_visible_values(causal):
    n, d = 17, 4
    v = rnd((n, d), 18)
    r = oracle.attention_head(rnd((n, d), 19), rnd((n, d), 20), v, 0.0, causal)
    for i in range(n):
        vis = i + 1 if causal else n
        np.testing.assert_allclose(r["o"][i], v[:vis].mean(axis=0), rtol=0, atol=1e-14)
        assert r["lse"][i] == pytest.approx(math.log(vis), abs=1e-14)


def test_causal_first_row_sees_only_first_key():
    n, d = 9, 3
    q, k, v = rnd((n, d), 21), rnd((n, d), 22), rnd((n, d), 23)
    r = oracle.attention_head(q, k, v, 1.1, True)
    np.testing.assert_allclose(r["o"][0], v[0], rtol=0, atol=0)
    # the last causal row equals the non-causal last row
    rn = oracle.attention_head(q, k, v, 1.1, False)
    np.testing.assert_allclose(r["o"][-1], rn["o"][-1], rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_changes_lse_by_row_constant_only(causal):
    n, d = 12, 6
    q, k, v = rnd((n, d), 24), rnd((n, d), 25), rnd((n, d), 26)
    c = rnd((d,), 27)
    a = oracle.attention_head(q, k, v, 0.6, causal)
    b = oracle.attention_head(q, k + c, v, 0.6, causal)
    np.testing.assert_allclose(b["o"], a["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(b["lse"] - a["lse"], 0.6 * (q @ c), rtol=0, atol=1e-13)


def test_scale_is_applied_to_scores():
    """Doubling the scale equals doubling Q (and differs from scale 1)."""
    n, d = 10, 4
    q, k, v = rnd((n, d), 28), rnd((n, d), 29), rnd((n, d), 30)
    a = oracle.attention_head(q, k, v, 2.0, False)
    b = oracle.attention_head(2.0 * q, k, v, 1.0, False)
    np.testing.assert_allclose(a["o"], b["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=0, atol=1e-13)
    c = oracle.attention_head(q, k, v, 1.0, False)
    assert np.abs(a["o"] - c["o"]).max() > 1e-3


def test_permutation_equivariance_non_causal():
    """Non-causal attention does not depend on key order, and permuting the
    queries permutes the output rows."""
    n, d = 15, 3
    q, k, v = rnd((n, d), 31), rnd((n, d), 32), rnd((n, d), 33)
    perm = np.random.default_rng(34).permutation(n)
    a = oracle.attention_head(q, k, v, 0.8, False)
    b = oracle.attention_head(q[perm], k[perm], v[perm], 0.8, False)
    np.testing.assert_allclose(b["o"], a["o"][perm], rtol=0, atol=1e-13)
    np.testing.assert_allclose(b["lse"], a["lse"][perm], rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# A library routine: PyTorch's scaled_dot_product_attention in float64
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 4), (19, 8), (64, 16)])
def test_matches_torch_sdpa_float64_forward_and_gradients(n, d, causal):
    q, k, v, do = (rnd((n, d), s) for s in (40, 41, 42, 43))
    scale = 1.0 / math.sqrt(d)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=scale)[0, 0]
    out.backward(torch.tensor(do))
    r = oracle.attention_head(q, k, v, scale, causal, dout=do)
    np.testing.assert_allclose(r["o"], out.detach().numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["dq"], tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dk"], tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dv"], tv.grad.numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Gradients: central finite differences of L = sum(dO * O)
# (mirrors the page's gradcheck in float64, l189.com walkthrough sec. 3.3)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 2), (4, 3), (8, 4)])
def test_gradients_by_central_differences(n, d, causal):
    q, k, v, do = rnd((n, d), 50), rnd((n, d), 51), rnd((n, d), 52), rnd((n, d), 53)
    scale, h = 0.7, 1e-6
    r = oracle.attention_head(q, k, v, scale, causal, dout=do)

    def loss(qq, kk, vv):
        return float((oracle.attention_head(qq, kk, vv, scale, causal)["o"] * do).sum())

    for name, arr, grad in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = plus, minus
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                       - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        err = np.abs(fd - grad).max() / max(np.abs(grad).max(), 1e-3)
        assert err <= 1e-6, (name, err)


# --------------------------------------------------------------------------
# Gradient identities and invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants_and_di_identity(causal):
    n, d = 48, 8
    q, k, v, do = (rnd((n, d), s) for s in (60, 61, 62, 63))
    r = oracle.attention_head(q, k, v, 0.35, causal, dout=do)
    # Di = sum_j P_ij dP_ij equals dO_i . O_i
    np.testing.assert_allclose(r["di"], (do * r["o"]).sum(axis=1), rtol=0, atol=1e-13)
    # sum_j dS_ij = 0  =>  sum_j dK_j = 0
    np.testing.assert_allclose(r["dk"].sum(axis=0), 0.0, rtol=0, atol=1e-12)
    # sum_j P_ij = 1  =>  sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(r["dv"].sum(axis=0), do.sum(axis=0), rtol=0, atol=1e-12)
    # dQ with V = const is zero (softmax of a constant output has no gradient)
    rc = oracle.attention_head(q, k, np.ones((n, d)), 0.35, causal, dout=do)
    np.testing.assert_allclose(rc["dq"], 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(rc["dk"], 0.0, rtol=0, atol=1e-12)


def test_value_gradient_is_linear_in_grad_output():
    n, d = 20, 4
    q, k, v = rnd((n, d), 64), rnd((n, d), 65), rnd((n, d), 66)
    do1, do2 = rnd((n, d), 67), rnd((n, d), 68)
    a = oracle.attention_head(q, k, v, 0.5, True, dout=do1)
    b = oracle.attention_head(q, k, v, 0.5, True, dout=do2)
    c = oracle.attention_head(q, k, v, 0.5, True, dout=do1 + 2 * do2)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(c[key], a[key] + 2 * b[key], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Sampled rows run the same code as the full call
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_full_rows_exactly(causal):
    n, d = 90, 8
    q, k, v, do = (rnd((n, d), s) for s in (70, 71, 72, 73))
    full = oracle.attention_head(q, k, v, 0.4, causal, dout=do)
    rows = np.array([0, 3, 17, 44, 89])
    part = oracle.attention_head(q, k, v, 0.4, causal, dout=do, rows=rows)
    for key in ("o", "lse", "dq", "di"):
        assert np.array_equal(part[key], full[key][rows]), key


def test_causal_tail_rows_give_exact_tail_key_gradients():
    n, d, t = 96, 8, 32
    q, k, v, do = (rnd((n, d), s) for s in (74, 75, 76, 77))
    full = oracle.attention_head(q, k, v, 0.4, True, dout=do)
    tail = np.arange(n - t, n)
    part = oracle.attention_head(q, k, v, 0.4, True, dout=do, rows=tail, kv_range=(n - t, n))
    np.testing.assert_allclose(part["dk"], full["dk"][n - t:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(part["dv"], full["dv"][n - t:], rtol=0, atol=1e-13)


def test_batched_wrapper_matches_per_head_calls():
    B, H, n, d = 2, 3, 10, 4
    q, k, v, do = (rnd((B, H, n, d), s) for s in (80, 81, 82, 83))
    res = oracle.attention(q, k, v, 0.5, True, dout=do)
    for b in range(B):
        for h in range(H):
            one = oracle.attention_head(q[b, h], k[b, h], v[b, h], 0.5, True, dout=do[b, h])
            for key in ("o", "lse", "dq", "dk", "dv"):
                assert np.array_equal(res[key][b, h], one[key])


def test_rejects_bad_arguments():
    q = np.zeros((4, 2))
    with pytest.raises(RuntimeError):
        oracle.attention_head(q, q, q, 1.0, False, rows=[7])
    with pytest.raises(ValueError):
        oracle.attention_head(q, np.zeros((5, 2)), q, 1.0, False)


def test_large_scores_concentrate_on_the_argmax_without_overflow():
    """Scores far beyond exp's range: the max shift (l189.com walkthrough,
    sec. 5.2) keeps everything finite, and softmax becomes one-hot at the
    largest score, so O_i = V_argmax and LSE_i = max_j S_ij."""
    n, d = 8, 3
    q = np.zeros((n, d))
    q[:, 0] = 1.0
    k = np.zeros((n, d))
    k[:, 0] = np.array([5.0, 900.0, -3.0, 2000.0, 1.0, 1500.0, 7.0, 0.0])
    v = rnd((n, d), 90)
    r = oracle.attention_head(q, k, v, 1.0, False)
    assert np.all(np.isfinite(r["o"])) and np.all(np.isfinite(r["lse"]))
    np.testing.assert_allclose(r["o"], np.tile(v[3], (n, 1)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["lse"], 2000.0, rtol=0, atol=1e-12)
    rc = oracle.attention_head(q, k, v, 1.0, True)
    # causal row 1 sees keys 0 and 1 only: the argmax there is key 1
    np.testing.assert_allclose(rc["o"][1], v[1], rtol=0, atol=1e-15)
    assert rc["lse"][1] == pytest.approx(900.0, abs=1e-12)


# --------------------------------------------------------------------------
# Sliding window and ALiBi (claire-chang.com FlashAttention introduction,
# flash_attn_func: window_size = (left, right), query i sees keys
# i - left .. i + right inclusive, -1 meaning no bound; alibi_slopes adds
# -slope * |i - j| to the score of query i and key j)
# --------------------------------------------------------------------------

def brute_force_banded(q, k, v, scale, causal, left, right, slope):
    """The definition with math.exp, written apart from the oracle."""
    n, d = q.shape
    o = np.zeros((n, d))
    lse = np.zeros(n)
    for i in range(n):
        s = []
        for j in range(n):
            if causal and j > i:
                continue
            if left != -1 and j < i - left:
                continue
            if right != -1 and j > i + right:
                continue
            s.append((j, scale * sum(q[i, t] * k[j, t] for t in range(d)) - slope * abs(i - j)))
        z = sum(math.exp(val) for _, val in s)
        lse[i] = math.log(z)
        for j, val in s:
            for t in range(d):
                o[i, t] += math.exp(val) / z * v[j, t]
    return o, lse


BANDS = [(-1, -1, 0.0), (2, 1, 0.0), (0, 0, 0.0), (3, -1, 0.0), (-1, 2, 0.0),
         (-1, -1, 0.5), (2, 3, 0.25), (1, -1, 1.5)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("left,right,slope", BANDS)
def test_window_and_alibi_brute_force(left, right, slope, causal):
    n, d = 7, 3
    q, k, v = rnd((n, d), 70), rnd((n, d), 71), rnd((n, d), 72)
    o_bf, lse_bf = brute_force_banded(q, k, v, 0.8, causal, left, right, slope)
    r = oracle.attention_head(q, k, v, 0.8, causal, window=(left, right), alibi_slope=slope)
    np.testing.assert_allclose(r["o"], o_bf, rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["lse"], lse_bf, rtol=0, atol=1e-13)


def additive_mask(n, causal, left, right, slope):
    """[n, n] float64 mask for torch SDPA: the ALiBi bias where visible,
    -inf elsewhere."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    ok = np.ones((n, n), bool)
    if causal:
        ok &= j <= i
    if left != -1:
        ok &= j >= i - left
    if right != -1:
        ok &= j <= i + right
    return np.where(ok, -slope * np.abs(i - j), -np.inf)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("left,right,slope", [(5, 3, 0.0), (-1, -1, 0.3), (4, 0, 0.7),
                                              (0, 6, 0.1)])
def test_window_and_alibi_match_torch_sdpa_float64(left, right, slope, causal):
    n, d = 23, 8
    q, k, v, do = (rnd((n, d), s) for s in (80, 81, 82, 83))
    scale = 1.0 / math.sqrt(d)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    mask = torch.tensor(additive_mask(n, causal, left, right, slope))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=mask[None, None],
        scale=scale)[0, 0]
    out.backward(torch.tensor(do))
    r = oracle.attention_head(q, k, v, scale, causal, dout=do, window=(left, right),
                              alibi_slope=slope)
    np.testing.assert_allclose(r["o"], out.detach().numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["dq"], tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dk"], tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dv"], tv.grad.numpy(), rtol=0, atol=1e-12)


def test_window_zero_is_the_identity_map():
    """window (0, 0): each query sees only its own key, so O = V and
    LSE_i = scale * Q_i . K_i."""
    n, d = 9, 4
    q, k, v = rnd((n, d), 90), rnd((n, d), 91), rnd((n, d), 92)
    r = oracle.attention_head(q, k, v, 0.6, False, window=(0, 0))
    np.testing.assert_allclose(r["o"], v, rtol=0, atol=1e-14)
    np.testing.assert_allclose(r["lse"], 0.6 * (q * k).sum(1), rtol=0, atol=1e-13)


def test_causal_equals_window_with_no_right_reach():
    n, d = 12, 4
    q, k, v, do = (rnd((n, d), s) for s in (93, 94, 95, 96))
    a = oracle.attention_head(q, k, v, 0.5, True, dout=do)
    b = oracle.attention_head(q, k, v, 0.5, False, dout=do, window=(-1, 0))
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(a[key], b[key], rtol=0, atol=1e-14)


def test_alibi_at_zero_scale_is_a_closed_form():
    """scale = 0 leaves only the bias: P_ij is proportional to exp(-slope |i-j|)
    and LSE_i = ln sum_j exp(-slope |i - j|)."""
    n, d, slope = 6, 3, 0.9
    q, k, v = rnd((n, d), 97), rnd((n, d), 98), rnd((n, d), 99)
    r = oracle.attention_head(q, k, v, 0.0, False, alibi_slope=slope)
    for i in range(n):
        w = np.array([math.exp(-slope * abs(i - j)) for j in range(n)])
        np.testing.assert_allclose(r["lse"][i], math.log(w.sum()), rtol=0, atol=1e-14)
        np.testing.assert_allclose(r["o"][i], (w / w.sum()) @ v, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_window_and_alibi_gradients_by_central_differences(causal):
    n, d = 6, 3
    q, k, v, do = rnd((n, d), 100), rnd((n, d), 101), rnd((n, d), 102), rnd((n, d), 103)
    scale, h, win, slope = 0.7, 1e-6, (2, 1), 0.4
    r = oracle.attention_head(q, k, v, scale, causal, dout=do, window=win, alibi_slope=slope)

    def loss(q, k, v):
        o = oracle.attention_head(q, k, v, scale, causal, window=win, alibi_slope=slope)["o"]
        return float((o * do).sum())

    for name, arr, grad in (("q", q, r["dq"]), ("k", k, r["dk"]), ("v", v, r["dv"])):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name] = arr.copy()
            args_m[name] = arr.copy()
            args_p[name][idx] += h
            args_m[name][idx] -= h
            fd[idx] = (loss(**args_p) - loss(**args_m)) / (2 * h)
        err = np.abs(fd - grad).max() / max(np.abs(grad).max(), 1e-3)
        assert err <= 1e-6, (name, err)


def test_batched_alibi_slopes_are_per_head_or_per_batch_and_head():
    B, H, n, d = 2, 3, 5, 2
    x = [rnd((B, H, n, d), s) for s in (104, 105, 106)]
    per_head = np.array([0.1, 0.5, 1.0])
    a = oracle.attention(*x, 0.5, False, alibi_slopes=per_head)
    b = oracle.attention(*x, 0.5, False, alibi_slopes=np.tile(per_head, (B, 1)))
    np.testing.assert_array_equal(a["o"], b["o"])
    for bb in range(B):
        for hh in range(H):
            one = oracle.attention_head(x[0][bb, hh], x[1][bb, hh], x[2][bb, hh], 0.5, False,
                                        alibi_slope=per_head[hh])
            np.testing.assert_array_equal(a["o"][bb, hh], one["o"])


def test_window_bounds_below_minus_one_are_rejected():
    q = rnd((4, 2), 107)
    with pytest.raises(RuntimeError):
        oracle.attention_head(q, q, q, 0.5, False, window=(-2, 0))


# --------------------------------------------------------------------------
# Block-sparse attention (the FlashAttention paper's block-sparse extension,
# as the pages report it): scores outside the blocks a mask keeps are -inf
# --------------------------------------------------------------------------

def brute_force_blocks(q, k, v, scale, causal, mask, T):
    """The definition with math.exp and an explicit block test; rows that see
    nothing give O = 0 and LSE = -inf."""
    n, d = q.shape
    o = np.zeros((n, d))
    lse = np.full(n, -np.inf)
    for i in range(n):
        s = [(j, scale * sum(q[i, t] * k[j, t] for t in range(d)))
             for j in range(n) if (not causal or j <= i) and mask[i // T][j // T]]
        if not s:
            continue
        z = sum(math.exp(val) for _, val in s)
        lse[i] = math.log(z)
        for j, val in s:
            for t in range(d):
                o[i, t] += math.exp(val) / z * v[j, t]
    return o, lse


def random_block_mask(nb, seed, density=0.5):
    m = (np.random.default_rng(seed).random((nb, nb)) < density).astype(np.uint8)
    return m


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,T,seed", [(7, 2, 1), (9, 3, 2), (8, 4, 3), (10, 3, 4)])
def test_block_mask_brute_force(n, T, seed, causal):
    d = 3
    q, k, v = rnd((n, d), 110 + seed), rnd((n, d), 111 + seed), rnd((n, d), 112 + seed)
    nb = (n + T - 1) // T
    mask = random_block_mask(nb, seed)
    o_bf, lse_bf = brute_force_blocks(q, k, v, 0.8, causal, mask, T)
    r = oracle.attention_head(q, k, v, 0.8, causal, block_mask=mask, block=T)
    np.testing.assert_allclose(r["o"], o_bf, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(r["lse"]), np.isinf(lse_bf))
    fin = np.isfinite(lse_bf)
    np.testing.assert_allclose(r["lse"][fin], lse_bf[fin], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_matches_torch_sdpa_float64(causal):
    """A mask that keeps every block row non-empty, against SDPA with the
    block mask expanded to an additive -inf mask."""
    n, d, T = 24, 8, 4
    nb = n // T
    mask = random_block_mask(nb, 7, 0.6)
    np.fill_diagonal(mask, 1)
    q, k, v, do = (rnd((n, d), s) for s in (120, 121, 122, 123))
    scale = 1.0 / math.sqrt(d)
    dense = np.kron(mask, np.ones((T, T))) > 0
    if causal:
        dense &= np.tril(np.ones((n, n), bool))
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    am = torch.tensor(np.where(dense, 0.0, -np.inf))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=am[None, None],
        scale=scale)[0, 0]
    out.backward(torch.tensor(do))
    r = oracle.attention_head(q, k, v, scale, causal, dout=do, block_mask=mask, block=T)
    np.testing.assert_allclose(r["o"], out.detach().numpy(), rtol=0, atol=1e-13)
    for name, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        np.testing.assert_allclose(r[name], t.grad.numpy(), rtol=0, atol=1e-12)


def test_block_diagonal_mask_is_attention_within_each_block():
    n, d, T = 12, 4, 4
    q, k, v, do = (rnd((n, d), s) for s in (124, 125, 126, 127))
    r = oracle.attention_head(q, k, v, 0.6, False, dout=do, block_mask=np.eye(3), block=T)
    for b in range(3):
        sl = slice(b * T, (b + 1) * T)
        one = oracle.attention_head(q[sl], k[sl], v[sl], 0.6, False, dout=do[sl])
        for key in ("o", "lse", "dq", "dk", "dv"):
            np.testing.assert_allclose(r[key][sl], one[key], rtol=0, atol=1e-14)


def test_rows_that_see_no_key_are_zero_and_carry_no_gradient():
    n, d, T = 8, 3, 4
    q, k, v, do = (rnd((n, d), s) for s in (128, 129, 130, 131))
    mask = np.array([[0, 0], [1, 1]])           # block row 0 sees nothing
    r = oracle.attention_head(q, k, v, 0.7, False, dout=do, block_mask=mask, block=T)
    assert np.all(r["o"][:4] == 0) and np.all(np.isneginf(r["lse"][:4]))
    assert np.all(r["dq"][:4] == 0)
    # the empty rows' dO does not reach dK, dV
    do2 = do.copy()
    do2[:4] += 5.0
    r2 = oracle.attention_head(q, k, v, 0.7, False, dout=do2, block_mask=mask, block=T)
    np.testing.assert_allclose(r2["dk"], r["dk"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r2["dv"], r["dv"], rtol=0, atol=1e-14)


def test_all_ones_block_mask_equals_no_mask():
    n, d = 11, 4
    q, k, v, do = (rnd((n, d), s) for s in (132, 133, 134, 135))
    a = oracle.attention_head(q, k, v, 0.5, True, dout=do)
    b = oracle.attention_head(q, k, v, 0.5, True, dout=do, block_mask=np.ones((4, 4)), block=3)
    for key in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[key], b[key])
