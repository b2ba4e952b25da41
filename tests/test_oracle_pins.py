"""Pins for the CPU float64 oracle: values fixed by the mathematics and by the
pages, none of them produced by the oracle itself.

Each test is chosen so that a plausible slip in the oracle (a dropped one-hot
term, a wrong sign or index, a transposed product, a missing 1/n, an unstable
log-sum-exp, wrong handling of ignored tokens) fails at least one of them.
"""
import json
import math
import os

import mpmath
import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(seed, N, D, V, scale=1.0):
    g = np.random.default_rng(seed)
    H = g.standard_normal((N, D))
    W = g.standard_normal((V, D)) * scale
    y = g.integers(0, V, N)
    return H, W, y


# ---- closed forms --------------------------------------------------------------

def test_zero_weights_closed_form():
    """W = 0: every logit is 0, lse = log V, loss = log V, dH = 0 and
    dW_v = sum_valid (1/V - [y_i = v]) h_i / n."""
    N, D, V = 7, 5, 11
    g = np.random.default_rng(1)
    H = g.standard_normal((N, D))
    W = np.zeros((V, D))
    y = np.array([3, -100, 0, 10, 3, -100, 7])
    r = oracle.flce(H, W, y)
    n = 5
    assert r["n_valid"] == n
    assert np.all(r["lse"] == math.log(V))
    assert r["loss"] == pytest.approx(math.log(V), rel=0, abs=1e-15)
    assert np.all(r["dH"] == 0.0)
    expect = np.zeros((V, D))
    for i in range(N):
        if y[i] == -100:
            continue
        expect += H[i][None, :] / V / n
        expect[y[i]] -= H[i] / n
    np.testing.assert_allclose(r["dW"], expect, rtol=0, atol=1e-15)


def test_two_class_logistic_closed_form():
    """V = 2 is binary logistic regression on the logit difference
    d_i = z_i1 - z_i0: loss_i = softplus(d_i) for label 0 and softplus(-d_i)
    for label 1; dL/dd_i = sigmoid(d_i) - [y_i = 1]."""
    N, D = 4, 3
    g = np.random.default_rng(2)
    H = g.standard_normal((N, D))
    W = g.standard_normal((2, D))
    y = np.array([0, 1, 1, 0])
    r = oracle.flce(H, W, y)
    d = H @ (W[1] - W[0])
    sig = 1.0 / (1.0 + np.exp(-d))
    per = np.where(y == 0, np.log1p(np.exp(d)), np.log1p(np.exp(-d)))
    assert r["loss"] == pytest.approx(per.mean(), rel=1e-14)
    t = (sig - (y == 1)) / N                        # dL/dd_i
    np.testing.assert_allclose(r["dH"], t[:, None] * (W[1] - W[0])[None, :], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r["dW"][1], (t[:, None] * H).sum(0), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r["dW"][0], -(t[:, None] * H).sum(0), rtol=1e-12, atol=1e-15)


def test_identical_rows_uniform_softmax():
    """All w_v equal: the softmax is uniform, so loss = log V whatever H is,
    and every gradient row of dL/dz is 1/V - onehot."""
    N, D, V = 5, 4, 9
    g = np.random.default_rng(3)
    H = g.standard_normal((N, D)) * 3
    w = g.standard_normal(D)
    W = np.tile(w, (V, 1))
    y = g.integers(0, V, N)
    r = oracle.flce(H, W, y)
    assert r["loss"] == pytest.approx(math.log(V), rel=1e-13)
    # dH_i = sum_v (1/V - [v=y_i]) w / N = 0 because every w_v is the same w.
    np.testing.assert_allclose(r["dH"], 0.0, atol=1e-14)


# ---- brute force ------------------------------------------------------------------

@pytest.mark.parametrize("shift", [0.0, 700.0, -745.0])
def test_lse_against_arbitrary_precision(shift):
    """The stable LSE equals log(sum exp z) evaluated with 50-digit arithmetic,
    including logits where exp(z) overflows or underflows a double."""
    g = np.random.default_rng(4)
    Z = g.standard_normal((6, 40)) * 5 + shift
    got = oracle.log_sum_exp_rows(Z)
    mpmath.mp.dps = 50
    for i in range(Z.shape[0]):
        exact = mpmath.log(mpmath.fsum(mpmath.exp(mpmath.mpf(float(z))) for z in Z[i]))
        assert float(exact) == pytest.approx(got[i], rel=1e-14, abs=1e-12)


def test_loss_against_arbitrary_precision():
    """Tiny case: the whole forward against a 50-digit evaluation of the definition."""
    N, D, V = 3, 4, 6
    H, W, y = _rand(5, N, D, V, scale=2.0)
    y[1] = -100
    r = oracle.flce(H, W, y)
    mpmath.mp.dps = 50
    tot = mpmath.mpf(0)
    n = 0
    for i in range(N):
        z = [mpmath.fsum(mpmath.mpf(float(H[i, d])) * mpmath.mpf(float(W[v, d])) for d in range(D))
             for v in range(V)]
        lse = mpmath.log(mpmath.fsum(mpmath.exp(t) for t in z))
        assert float(lse) == pytest.approx(r["lse"][i], rel=1e-14)
        if y[i] != -100:
            tot += lse - z[y[i]]
            n += 1
    assert float(tot / n) == pytest.approx(r["loss"], rel=1e-14)


# ---- finite differences ------------------------------------------------------------

@pytest.mark.parametrize("reduction,grad_scale", [("mean", 1.0), ("sum", 1.0), ("mean", 0.37)])
def test_gradients_central_differences(reduction, grad_scale):
    N, D, V = 4, 6, 5
    H, W, y = _rand(6, N, D, V)
    y[2] = -100
    r = oracle.flce(H, W, y, reduction=reduction, grad_scale=grad_scale)

    def f(Hx, Wx):
        return grad_scale * oracle.flce(Hx, Wx, y, reduction=reduction, want_grads=False)["loss"]

    h = 1e-6
    num_dH = np.zeros_like(H)
    for i in range(N):
        for d in range(D):
            Hp, Hm = H.copy(), H.copy()
            Hp[i, d] += h
            Hm[i, d] -= h
            num_dH[i, d] = (f(Hp, W) - f(Hm, W)) / (2 * h)
    num_dW = np.zeros_like(W)
    for v in range(V):
        for d in range(D):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, d] += h
            Wm[v, d] -= h
            num_dW[v, d] = (f(H, Wp) - f(H, Wm)) / (2 * h)
    np.testing.assert_allclose(r["dH"], num_dH, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(r["dW"], num_dW, rtol=1e-6, atol=1e-8)
    assert np.all(r["dH"][2] == 0.0)


def test_gradients_central_differences_square():
    """N = V = D, so a transposed product would still have the right shape."""
    N = D = V = 5
    H, W, y = _rand(7, N, D, V)
    r = oracle.flce(H, W, y)

    def f(Hx, Wx):
        return oracle.flce(Hx, Wx, y, want_grads=False)["loss"]

    h = 1e-6
    for (i, d) in [(0, 1), (3, 4), (4, 0)]:
        Hp, Hm = H.copy(), H.copy()
        Hp[i, d] += h
        Hm[i, d] -= h
        assert r["dH"][i, d] == pytest.approx((f(Hp, W) - f(Hm, W)) / (2 * h), rel=1e-6, abs=1e-9)
        Wp, Wm = W.copy(), W.copy()
        Wp[i, d] += h
        Wm[i, d] -= h
        assert r["dW"][i, d] == pytest.approx((f(H, Wp) - f(H, Wm)) / (2 * h), rel=1e-6, abs=1e-9)


# ---- invariants --------------------------------------------------------------------

def test_dlogits_rows_sum_to_zero():
    """sum_v g_iv = 0 for every token, hence sum_v dW_v = sum_i (sum_v g_iv) h_i = 0."""
    H, W, y = _rand(8, 9, 7, 13)
    r = oracle.flce(H, W, y)
    np.testing.assert_allclose(r["dW"].sum(axis=0), 0.0, atol=1e-15)


def test_ignored_token_equals_removed_token_with_same_n():
    """An ignored token changes nothing but is not counted: the loss and dW
    equal those of the batch without it, and its dH row is exactly zero."""
    H, W, y = _rand(9, 6, 5, 8)
    y2 = y.copy()
    y2[4] = -100
    r = oracle.flce(H, W, y2)
    keep = [0, 1, 2, 3, 5]
    r2 = oracle.flce(H[keep], W, y[keep])
    assert r["n_valid"] == 5
    assert r["loss"] == pytest.approx(r2["loss"], rel=1e-14)
    np.testing.assert_allclose(r["dW"], r2["dW"], rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(r["dH"][keep], r2["dH"], rtol=1e-13, atol=1e-16)
    assert np.all(r["dH"][4] == 0.0)
    assert r["nll"][4] == 0.0
    # lse is still written for the ignored token
    assert r["lse"][4] == pytest.approx(oracle.log_sum_exp_rows(H[4:5] @ W.T)[0], rel=1e-15)


def test_shift_invariance():
    """Adding the same vector c to every w_v adds h_i.c to every logit of row i,
    which leaves softmax, loss and dH unchanged."""
    H, W, y = _rand(10, 6, 5, 9)
    c = np.random.default_rng(11).standard_normal(5)
    r = oracle.flce(H, W, y)
    r2 = oracle.flce(H, W + c[None, :], y)
    assert r2["loss"] == pytest.approx(r["loss"], rel=1e-12)
    np.testing.assert_allclose(r2["dH"], r["dH"], rtol=1e-10, atol=1e-14)


def test_permutation_equivariance():
    H, W, y = _rand(12, 8, 5, 10)
    g = np.random.default_rng(13)
    pt = g.permutation(8)
    pv = g.permutation(10)
    inv_pv = np.argsort(pv)
    r = oracle.flce(H, W, y)
    r2 = oracle.flce(H[pt], W[pv], inv_pv[y[pt]])
    assert r2["loss"] == pytest.approx(r["loss"], rel=1e-13)
    np.testing.assert_allclose(r2["dH"], r["dH"][pt], rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(r2["dW"], r["dW"][pv], rtol=1e-12, atol=1e-16)


def test_reductions_and_scales():
    H, W, y = _rand(14, 6, 4, 7)
    y[0] = -100
    m = oracle.flce(H, W, y)
    s = oracle.flce(H, W, y, reduction="sum")
    assert s["loss"] == pytest.approx(m["loss"] * 5, rel=1e-14)
    np.testing.assert_allclose(s["dW"], m["dW"] * 5, rtol=1e-13)
    g = oracle.flce(H, W, y, grad_scale=2.5)
    np.testing.assert_allclose(g["dH"], m["dH"] * 2.5, rtol=1e-13)
    assert g["loss"] == pytest.approx(m["loss"], rel=1e-15)
    z = oracle.flce(H, W, y, normalizer=20.0)
    assert z["loss"] == pytest.approx(m["loss"] * 5 / 20, rel=1e-14)
    np.testing.assert_allclose(z["dW"], m["dW"] * 5 / 20, rtol=1e-13)


def test_all_ignored_gives_zero_loss_and_gradients():
    H, W, y = _rand(15, 4, 3, 5)
    y[:] = -100
    r = oracle.flce(H, W, y)
    assert r["n_valid"] == 0 and r["loss"] == 0.0
    assert np.all(r["dH"] == 0) and np.all(r["dW"] == 0)
    assert np.all(np.isfinite(r["lse"]))


def test_out_of_range_label_is_rejected():
    H, W, y = _rand(16, 4, 3, 5)
    for bad in (5, -1, -101):
        yy = y.copy()
        yy[2] = bad
        with pytest.raises(ValueError):
            oracle.flce(H, W, yy)


def test_selected_rows_match_full():
    H, W, y = _rand(17, 40, 8, 30)
    y[[3, 9]] = -100
    full = oracle.flce(H, W, y, row_block=7, vocab_block=4)
    rows = np.array([0, 3, 17, 39])
    vids = np.array([1, 2, 29])
    part = oracle.flce(H, W, y, dh_rows=rows, dw_rows=vids)
    np.testing.assert_array_equal(part["dH"], full["dH"][rows])
    np.testing.assert_allclose(part["dW"], full["dW"][vids], rtol=1e-14, atol=1e-17)
    np.testing.assert_array_equal(part["lse"], full["lse"])


def test_chunked_streaming_equals_unfused_on_the_pages_example():
    """The pages' simulation (section "Implementation: Simulating Fused Linear
    Cross-Entropy in Python") checks that processing tokens 16 at a time gives
    the same loss and dH as the full [N, V] computation, at N=128, D=512,
    V=4096 with numpy seed 42, H and W standard normal in float32. Here the
    token-chunked pass is written independently (16-token chunks, float64)
    and compared to the oracle."""
    N, D, V = 128, 512, 4096
    np.random.seed(42)
    H = np.random.randn(N, D).astype(np.float32)
    W = np.random.randn(V, D).astype(np.float32)
    y = np.random.randint(0, V, size=(N,))
    r = oracle.flce(H, W, y)
    Hd, Wd = H.astype(np.float64), W.astype(np.float64)
    total = 0.0
    dH = np.zeros((N, D))
    for i in range(0, N, 16):
        z = Hd[i:i + 16] @ Wd.T
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        s = e.sum(axis=1, keepdims=True)
        lse = np.log(s) + m
        k = np.arange(z.shape[0])
        total += float(np.sum(lse[:, 0] - z[k, y[i:i + 16]]))
        p = e / s
        p[k, y[i:i + 16]] -= 1.0
        dH[i:i + 16] = (p / N) @ Wd
    assert abs(total / N - r["loss"]) < 1e-9
    assert np.max(np.abs(dH - r["dH"])) < 1e-12


# ---- the pages' printed memory figures ---------------------------------------------

def test_logits_bytes_matches_printed_sizes():
    with open(os.path.join(GOLDEN, "logits_memory.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        got = oracle.logits_bytes(c["N"], c["V"]) / 1e9
        assert round(got, c["decimals"]) == pytest.approx(c["printed_GB"], abs=1e-12), c["citation"]


# ---- sampling helpers --------------------------------------------------------------

def test_sample_helpers_are_deterministic_and_cover_edge_ids():
    g = np.random.default_rng(18)
    y = g.integers(0, 1000, 5000)
    y[g.permutation(5000)[:100]] = -100
    a = oracle.sample_rows(y, 256, seed=0)
    b = oracle.sample_rows(y, 256, seed=0)
    np.testing.assert_array_equal(a, b)
    assert 200 <= len(a) <= 256 and np.all(np.diff(a) > 0)
    assert np.sum(y[a] == -100) >= 16
    v = oracle.sample_vocab(y, 1000, 64, seed=0)
    assert 999 in v and len(v) == 64 and np.all(np.diff(v) > 0)


# ---- cross-entropy over given logits ----------------------------------------------

def test_ce_logits_zero_logits_closed_form():
    """Z = 0: lse = log V for every token, loss = log V, dZ = (1/V - onehot)/n."""
    N, V = 6, 9
    y = np.array([0, 8, -100, 3, 3, 5])
    r = oracle.ce_logits(np.zeros((N, V)), y)
    assert np.all(r["lse"] == math.log(V))
    assert r["loss"] == pytest.approx(math.log(V), rel=1e-15)
    n = 5
    expect = np.full((N, V), 1.0 / V / n)
    expect[2] = 0.0
    for i, t in enumerate(y):
        if t != -100:
            expect[i, t] -= 1.0 / n
    np.testing.assert_allclose(r["dZ"], expect, rtol=0, atol=1e-16)


def test_ce_logits_two_class_closed_form():
    """V = 2: loss_i = softplus(z_other - z_target), dz_target = -sigmoid(z_other - z_target)/n."""
    Z = np.array([[0.3, -1.2], [2.0, 0.5], [-0.7, 0.4]])
    y = np.array([0, 1, 1])
    r = oracle.ce_logits(Z, y)
    d = np.array([Z[0, 1] - Z[0, 0], Z[1, 0] - Z[1, 1], Z[2, 0] - Z[2, 1]])
    assert r["loss"] == pytest.approx(np.log1p(np.exp(d)).mean(), rel=1e-14)
    sig = 1 / (1 + np.exp(-d))
    for i in range(3):
        assert r["dZ"][i, y[i]] == pytest.approx(-sig[i] / 3, rel=1e-13)
        assert r["dZ"][i, 1 - y[i]] == pytest.approx(sig[i] / 3, rel=1e-13)


def test_ce_logits_central_differences():
    g = np.random.default_rng(30)
    Z = g.standard_normal((4, 7)) * 3
    y = np.array([1, -100, 6, 0])
    r = oracle.ce_logits(Z, y, reduction="sum", grad_scale=0.5)
    h = 1e-6
    for i in range(4):
        for v in range(7):
            Zp, Zm = Z.copy(), Z.copy()
            Zp[i, v] += h
            Zm[i, v] -= h
            num = 0.5 * (oracle.ce_logits(Zp, y, reduction="sum", want_grad=False)["loss"] -
                         oracle.ce_logits(Zm, y, reduction="sum", want_grad=False)["loss"]) / (2 * h)
            assert r["dZ"][i, v] == pytest.approx(num, rel=1e-6, abs=1e-9)


def test_ce_logits_none_reduction_and_large_logits():
    """Per-token losses; logits near 800 where exp overflows a double."""
    Z = np.array([[800.0, 799.0, 790.0], [-750.0, -760.0, -751.0]])
    y = np.array([1, -100])
    r = oracle.ce_logits(Z, y, reduction="none")
    mpmath.mp.dps = 50
    exact = mpmath.log(mpmath.fsum(mpmath.exp(mpmath.mpf(z)) for z in Z[0])) - 799
    assert r["loss"][0] == pytest.approx(float(exact), rel=1e-14)
    assert r["loss"][1] == 0.0 and r["dZ"] is None


def test_gradient_operands_enter_only_the_two_products():
    """With Hg, Wg given, the loss and lse still come from H, W, and the
    gradients are the same G times the substituted operands."""
    H, W, y = _rand(31, 6, 5, 9)
    g = np.random.default_rng(32)
    Hg = H + g.standard_normal(H.shape) * 0.1
    Wg = W * 0.5
    a = oracle.flce(H, W, y)
    b = oracle.flce(H, W, y, Hg=Hg, Wg=Wg)
    assert b["loss"] == a["loss"]
    np.testing.assert_array_equal(b["lse"], a["lse"])
    np.testing.assert_allclose(b["dH"], a["dH"] * 0.5, rtol=1e-13, atol=1e-16)
    # dW is linear in Hg: dW(Hg) - dW(H) = dW computed with (Hg - H)
    c = oracle.flce(H, W, y, Hg=Hg - H, Wg=W)
    np.testing.assert_allclose(b["dW"] - a["dW"], c["dW"], rtol=1e-10, atol=1e-14)


# ---- magnitude products (the rounding scale of each gradient element) ------------

def test_magnitude_products_zero_weights_closed_form():
    """W = 0: g_iv = (1/V - [y_i = v]) / n, so |G|^T |H| has the closed form
    sum_valid (|1/V - [y_i = v]| / n) |h_i| and |G| |W| = 0."""
    N, D, V = 7, 5, 11
    g = np.random.default_rng(41)
    H = g.standard_normal((N, D))
    y = np.array([3, -100, 0, 10, 3, -100, 7])
    r = oracle.flce(H, np.zeros((V, D)), y, want_abs=True)
    n = 5
    expect = np.zeros((V, D))
    for i in range(N):
        if y[i] == -100:
            continue
        for v in range(V):
            expect[v] += abs(1.0 / V - (1.0 if v == y[i] else 0.0)) / n * np.abs(H[i])
    np.testing.assert_allclose(r["dW_abs"], expect, rtol=0, atol=1e-15)
    assert np.all(r["dH_abs"] == 0.0)


def test_magnitude_products_brute_force():
    """Loops over the definition g_iv = (exp(z_iv - lse_i) - [v = y_i]) * scale with
    lse from mpmath, then sum_v |g_iv| |w_vd| and sum_i |g_iv| |h_id|; selected rows,
    ignored tokens and a gradient scale included."""
    N, D, V = 6, 4, 9
    H, W, y = _rand(42, N, D, V, scale=0.7)
    y[2] = -100
    rows, vids = np.array([0, 2, 5]), np.array([1, 4, 8])
    r = oracle.flce(H, W, y, grad_scale=0.3, dh_rows=rows, dw_rows=vids, want_abs=True)
    n = 5
    G = np.zeros((N, V))
    for i in range(N):
        if y[i] == -100:
            continue
        z = [sum(float(H[i, d]) * float(W[v, d]) for d in range(D)) for v in range(V)]
        lse = float(mpmath.log(mpmath.fsum(mpmath.exp(mpmath.mpf(t)) for t in z)))
        for v in range(V):
            G[i, v] = (math.exp(z[v] - lse) - (1.0 if v == y[i] else 0.0)) * 0.3 / n
    for k, i in enumerate(rows):
        for d in range(D):
            want = sum(abs(G[i, v]) * abs(W[v, d]) for v in range(V))
            assert r["dH_abs"][k, d] == pytest.approx(want, rel=1e-12, abs=1e-15)
    for k, v in enumerate(vids):
        for d in range(D):
            want = sum(abs(G[i, v]) * abs(H[i, d]) for i in range(N))
            assert r["dW_abs"][k, d] == pytest.approx(want, rel=1e-12, abs=1e-15)


def test_magnitude_products_bound_and_equal_the_signed_ones_without_cancellation():
    """|dH| <= |G||W| and |dW| <= |G|^T|H| everywhere (triangle inequality), with
    equality for the dW row of an id that no token has as its label when H >= 0
    (every g_iv of that column is then positive, so nothing cancels)."""
    N, D, V = 40, 16, 30
    H, W, y = _rand(43, N, D, V, scale=0.5)
    H = np.abs(H)
    y = np.where(y == 7, 8, y)   # id 7: no hits
    y[::9] = -100
    r = oracle.flce(H, W, y, want_abs=True)
    assert np.all(np.abs(r["dH"]) <= r["dH_abs"] * (1 + 1e-12))
    assert np.all(np.abs(r["dW"]) <= r["dW_abs"] * (1 + 1e-12))
    np.testing.assert_allclose(r["dW"][7], r["dW_abs"][7], rtol=1e-13, atol=0)
    assert np.all(r["dH_abs"][y == -100] == 0.0)
