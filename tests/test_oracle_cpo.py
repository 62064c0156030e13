"""Pins of the CPO oracle (page "Fused linear + CPO loss": x [batch, seq,
hidden], weight [vocab, hidden], target [batch, seq], loss [1]; the page names
the CPO objective without printing it, so the oracle takes the published one:
loss = alpha * NLL(chosen) + mean_pairs -ln sigmoid(beta (lp_chosen -
lp_rejected)), chosen = the first half of the batch).

The pins reach the oracle from outside its own code: closed forms (zero
activations, identical chosen and rejected answers, the large-margin limit),
the softplus identity under swapping the halves, a 40-digit brute force that
multiplies token probabilities instead of summing log-softmax terms, the NLL
against the separately pinned fused CE, and the gradient against central
differences of the forward."""
import math

import mpmath
import numpy as np
import pytest

import gen
import oracle


def rand_case(seed, B, S, H, V, sx=1.0, sw=0.5):
    x = gen.normal_f64(seed, 0, (B, S, H), sigma=sx)
    W = gen.normal_f64(seed, 1, (V, H), sigma=sw)
    t = gen.targets(seed, 2, (B, S), V)
    return x, W, t


@pytest.mark.parametrize("alpha", [0.0, 1.0, 2.5])
def test_zero_activations_closed_form(alpha):
    # every logit 0: each token loss is ln V, every margin 0, so
    # loss = alpha ln V + ln 2 and lp_b = -S ln V
    B, S, H, V = 6, 5, 8, 11
    W = gen.normal_f64(1, 1, (V, H))
    t = gen.targets(1, 2, (B, S), V)
    m, rows, lp = oracle.cpo_f64(np.zeros((B, S, H)), W, t, beta=0.3, alpha=alpha)
    assert m == pytest.approx(alpha * math.log(V) + math.log(2), rel=1e-14)
    np.testing.assert_allclose(rows, math.log(V), rtol=1e-14)
    np.testing.assert_allclose(lp, -S * math.log(V), rtol=1e-14)


def test_identical_answers_give_ln2_preference():
    # rejected sequence k = chosen sequence k (same activations and targets):
    # every margin is exactly 0, so loss - alpha * nll = ln 2 for any beta
    B, S, H, V = 4, 7, 16, 40
    x, W, t = rand_case(2, B, S, H, V)
    x[2:] = x[:2]
    t[2:] = t[:2]
    for beta in (0.1, 1.0, 7.0):
        m1, _, lp = oracle.cpo_f64(x, W, t, beta=beta, alpha=1.0)
        m0, _, _ = oracle.cpo_f64(x, W, t, beta=beta, alpha=0.0)
        assert np.array_equal(lp[:2], lp[2:])
        assert m0 == pytest.approx(math.log(2), rel=1e-15)
        assert m1 > m0


def test_nll_term_is_the_fused_ce_mean_of_the_chosen_half():
    B, S, H, V = 6, 4, 12, 30
    x, W, t = rand_case(3, B, S, H, V)
    m1, rows, _ = oracle.cpo_f64(x, W, t, beta=0.2, alpha=1.0)
    m2, _, _ = oracle.cpo_f64(x, W, t, beta=0.2, alpha=2.0)
    nll_ref, rows_ref = oracle.flce_f64(x[: B // 2].reshape(-1, H), W, t[: B // 2].reshape(-1))
    assert m2 - m1 == pytest.approx(nll_ref, rel=1e-12)
    np.testing.assert_allclose(rows[: B // 2].reshape(-1), rows_ref, rtol=1e-15)


def test_swapping_halves_follows_the_softplus_identity():
    # softplus(-u) - softplus(u) = -u: with the halves swapped every margin
    # changes sign, so pref' - pref = (beta / Bc) sum_k d_k
    B, S, H, V = 8, 3, 10, 25
    x, W, t = rand_case(4, B, S, H, V, sx=2.0)
    beta = 0.7
    m, _, lp = oracle.cpo_f64(x, W, t, beta=beta, alpha=0.0)
    xs = np.concatenate([x[B // 2:], x[: B // 2]])
    ts = np.concatenate([t[B // 2:], t[: B // 2]])
    ms, _, _ = oracle.cpo_f64(xs, W, ts, beta=beta, alpha=0.0)
    d = lp[: B // 2] - lp[B // 2:]
    assert abs(d).max() > 1.0                 # margins far from 0: a real test of the sign
    assert ms - m == pytest.approx(beta * d.sum() / (B // 2), rel=1e-12)


def test_large_margin_limit():
    # chosen answers far more likely than rejected ones: beta d ~ 60, so the
    # preference term is e^{-beta d} to within e^{-2 beta d}
    B, S, H, V = 2, 2, 4, 6
    W = np.eye(V, H) * 1.0
    W[4:] = 0.0
    x = np.zeros((B, S, H))
    t = np.zeros((B, S), np.int64)
    x[0, :, 0] = 40.0     # chosen: target 0 holds a logit of 40
    x[1, :, 1] = 40.0     # rejected: logit 40 on class 1, target still 0
    beta = 1.0
    m, _, lp = oracle.cpo_f64(x, W, t, beta=beta, alpha=0.0)
    d = lp[0] - lp[1]
    assert d > 60
    assert m == pytest.approx(math.exp(-beta * d), rel=1e-12)


def test_brute_force_probability_route():
    # -ln sigmoid(beta ln(P_w / P_l)) with P the product of token probabilities,
    # at 40 significant digits, on integer-valued activations and weights
    mpmath.mp.dps = 40
    rng = np.random.default_rng(7)
    B, S, H, V = 4, 2, 3, 4
    x = rng.integers(-2, 3, size=(B, S, H)).astype(np.float64)
    W = rng.integers(-2, 3, size=(V, H)).astype(np.float64)
    t = rng.integers(0, V, size=(B, S))
    beta, alpha = 0.5, 1.5
    m, _, lp = oracle.cpo_f64(x, W, t, beta=beta, alpha=alpha)
    P = []
    nll = mpmath.mpf(0)
    for b in range(B):
        prob = mpmath.mpf(1)
        for s in range(S):
            z = [mpmath.mpf(float(np.dot(x[b, s], W[v]))) for v in range(V)]
            p = mpmath.e ** z[t[b, s]] / mpmath.fsum(mpmath.e ** zv for zv in z)
            prob *= p
            if b < B // 2:
                nll -= mpmath.log(p)
        P.append(prob)
        assert lp[b] == pytest.approx(float(mpmath.log(prob)), rel=1e-13)
    pref = mpmath.fsum(-mpmath.log(1 / (1 + (P[k + B // 2] / P[k]) ** beta)) for k in range(B // 2))
    want = alpha * nll / (B // 2 * S) + pref / (B // 2)
    assert m == pytest.approx(float(want), rel=1e-13)


@pytest.mark.parametrize("beta,alpha", [(0.1, 1.0), (2.0, 0.0), (0.5, 3.0)])
def test_grads_match_central_differences(beta, alpha):
    B, S, H, V = 4, 3, 5, 7
    x, W, t = rand_case(5, B, S, H, V, sx=1.0, sw=0.8)
    scale = 1.5
    dx, dW = oracle.cpo_grad_f64(x, W, t, beta=beta, alpha=alpha, scale=scale)
    f = lambda xx, WW: scale * oracle.cpo_f64(xx, WW, t, beta=beta, alpha=alpha)[0]  # noqa: E731
    h = 1e-6
    for idx in [(0, 0, 0), (1, 2, 4), (2, 1, 3), (3, 0, 1), (3, 2, 2)]:
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        assert dx[idx] == pytest.approx((f(xp, W) - f(xm, W)) / (2 * h), rel=1e-6, abs=1e-10)
    for idx in [(0, 0), (3, 4), (6, 2), (5, 1)]:
        Wp, Wm = W.copy(), W.copy()
        Wp[idx] += h
        Wm[idx] -= h
        assert dW[idx] == pytest.approx((f(x, Wp) - f(x, Wm)) / (2 * h), rel=1e-6, abs=1e-10)


def test_bf16_front_end_and_bad_target():
    B, S, H, V = 2, 3, 16, 9
    x = gen.normal_bf16_bits(6, 0, (B, S, H))
    W = gen.normal_bf16_bits(6, 1, (V, H), sigma=0.5)
    t = gen.targets(6, 2, (B, S), V)
    m16, rows16, lp16 = oracle.cpo_bf16(x, W, t, beta=0.1, alpha=1.0)
    m64, rows64, lp64 = oracle.cpo_f64(gen.bf16_bits_to_f32(x).astype(np.float64),
                                       gen.bf16_bits_to_f32(W).astype(np.float64), t, beta=0.1, alpha=1.0)
    assert m16 == m64 and np.array_equal(rows16, rows64) and np.array_equal(lp16, lp64)
    g16 = oracle.cpo_grad_bf16(x, W, t)
    g64 = oracle.cpo_grad_f64(gen.bf16_bits_to_f32(x).astype(np.float64),
                              gen.bf16_bits_to_f32(W).astype(np.float64), t)
    assert np.array_equal(g16[0], g64[0]) and np.array_equal(g16[1], g64[1])
    t[1, 2] = -1
    m, rows, lp = oracle.cpo_bf16(x, W, t)
    assert math.isnan(m) and np.isnan(rows[1, 2]) and np.isnan(lp[1]) and np.isfinite(lp[0])


def test_combine_weights_are_the_derivative_of_the_combination():
    # d loss / d l_i by central differences of the combination itself, and the
    # combination of the oracle's own rows reproduces the full oracle
    B, S = 6, 4
    rng = np.random.default_rng(9)
    rows = rng.uniform(0.5, 6.0, size=(B, S))
    m, lp, w = oracle.cpo_combine(rows, beta=0.4, alpha=1.3)
    np.testing.assert_allclose(lp, -rows.sum(axis=1), rtol=1e-15)
    # loss ~ 4: fp64 round-off over 2h = 2e-5 is ~1e-10 and the h^2 term smaller
    h = 1e-5
    for i in range(B):
        for s in range(S):
            rp, rm = rows.copy(), rows.copy()
            rp[i, s] += h
            rm[i, s] -= h
            fd = (oracle.cpo_combine(rp, 0.4, 1.3)[0] - oracle.cpo_combine(rm, 0.4, 1.3)[0]) / (2 * h)
            assert w[i, s] == pytest.approx(fd, rel=1e-6, abs=1e-9)
    x, W, t = rand_case(8, B, S, 6, 10)
    mo, ro, lpo = oracle.cpo_f64(x, W, t, beta=0.4, alpha=1.3)
    mc, lpc, _ = oracle.cpo_combine(ro, 0.4, 1.3)
    assert mc == mo and np.array_equal(lpc, lpo)
