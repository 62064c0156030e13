"""Pins of the cross-entropy backward oracle (gradient of the losses of the
pages "Cross-entropy loss" and "Vocab-parallel cross-entropy, Megatron
layout" with respect to the logits): central finite differences of the
independently pinned forward oracle, zero row sums, closed forms."""
import math

import numpy as np
import pytest

import gen
import oracle


def test_matches_central_differences_of_the_forward():
    T, V = 3, 7
    z = gen.normal_f64(20, 0, (T, V), sigma=1.5)
    t = gen.targets(20, 1, (T,), V)
    dz = oracle.ce_grad_f64(z, t, None, scale=1.0 / T)   # gradient of the mean
    h = 1e-5
    for i in range(T):
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[i, v] += h
            zm[i, v] -= h
            fd = (oracle.ce_f64(zp, t)[0] - oracle.ce_f64(zm, t)[0]) / (2 * h)
            assert dz[i, v] == pytest.approx(fd, rel=1e-6, abs=1e-10)


def test_weighted_rows_match_central_differences():
    T, V = 4, 5
    z = gen.normal_f64(21, 0, (T, V))
    t = gen.targets(21, 1, (T,), V)
    w = np.array([0.5, -2.0, 0.0, 3.0])
    dz = oracle.ce_grad_f64(z, t, w, scale=2.0)
    h = 1e-5
    for i in range(T):
        for v in range(V):
            zp, zm = z.copy(), z.copy()
            zp[i, v] += h
            zm[i, v] -= h
            lp = oracle.ce_f64(zp, t)[1]
            lm = oracle.ce_f64(zm, t)[1]
            fd = 2.0 * np.dot(w, lp - lm) / (2 * h)
            assert dz[i, v] == pytest.approx(fd, rel=1e-6, abs=1e-10)


def test_rows_sum_to_zero_and_target_column_is_negative():
    z = gen.normal_f64(22, 0, (6, 300), sigma=3.0)
    t = gen.targets(22, 1, (6,), 300)
    dz = oracle.ce_grad_f64(z, t)
    np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-14)
    assert np.all(dz[np.arange(6), t] < 0)
    mask = np.ones_like(dz, bool)
    mask[np.arange(6), t] = False
    assert np.all(dz[mask] > 0)


def test_closed_forms():
    V = 9
    dz = oracle.ce_grad_f64(np.full((2, V), 4.0), np.array([0, 8]))
    want = np.full((2, V), 1.0 / V)
    want[0, 0] -= 1
    want[1, 8] -= 1
    np.testing.assert_allclose(dz, want, rtol=1e-14, atol=1e-16)
    assert np.all(oracle.ce_grad_f64(np.array([[2.5], [-1.0]]), np.array([0, 0])) == 0.0)


def test_bad_target_row_is_nan_and_flat_scale():
    z = gen.normal_f32(23, 0, (4, 50))
    t = gen.targets(23, 1, (4,), 50)
    t[2] = 50
    dz = oracle.ce_grad_f32(z, t, scale=3.0)
    assert np.all(np.isnan(dz[2])) and np.all(np.isfinite(np.delete(dz, 2, axis=0)))
    ref = oracle.ce_grad_f64(z.astype(np.float64)[[0, 1, 3]], t[[0, 1, 3]], scale=3.0 / 4)
    np.testing.assert_array_equal(np.delete(dz, 2, axis=0), ref)


def test_sbv_layout_uses_row_s_times_B_plus_b():
    S, B, V = 3, 2, 16
    zb = gen.normal_bf16_bits(24, 0, (S, B, V), sigma=2.0)
    t = gen.targets(24, 1, (S, B), V)
    dl = np.arange(1, S * B + 1, dtype=np.float64).reshape(S, B)
    dz = oracle.ce_grad_sbv_bf16(zb, t, dl, scale=0.5)
    z = gen.bf16_bits_to_f32(zb).astype(np.float64).reshape(S * B, V)
    ref = oracle.ce_grad_f64(z, t.reshape(-1), dl.reshape(-1), scale=0.5).reshape(S, B, V)
    np.testing.assert_array_equal(dz, ref)
    # weight k+1 on row k: row k's gradient is (k+1)/1 times row k's unit-weight gradient
    unit = oracle.ce_grad_sbv_bf16(zb, t, None, scale=1.0)
    np.testing.assert_allclose(dz, 0.5 * dl[:, :, None] * unit, rtol=1e-15)


# ---------------------------------------------------------------- fused linear + CE backward
def test_flce_f64_forward_matches_bf16_oracle():
    x = gen.normal_bf16_bits(25, 0, (4, 24))
    W = gen.normal_bf16_bits(25, 2, (31, 24), sigma=0.5)
    t = gen.targets(25, 1, (4,), 31)
    widen = lambda b: gen.bf16_bits_to_f32(b).astype(np.float64)  # noqa: E731
    a = oracle.flce_bf16(x, W, t)
    b = oracle.flce_f64(widen(x), widen(W), t)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


def test_flce_grads_match_central_differences():
    T, H, V = 3, 5, 7
    x = gen.normal_f64(26, 0, (T, H))
    W = gen.normal_f64(26, 2, (V, H), sigma=0.7)
    t = gen.targets(26, 1, (T,), V)
    scale = 1.3
    dx, dW = oracle.flce_grad_f64(x, W, t, scale)
    h = 1e-5
    for i in range(T):
        for k in range(H):
            xp, xm = x.copy(), x.copy()
            xp[i, k] += h
            xm[i, k] -= h
            fd = scale * (oracle.flce_f64(xp, W, t)[0] - oracle.flce_f64(xm, W, t)[0]) / (2 * h)
            assert dx[i, k] == pytest.approx(fd, rel=1e-6, abs=1e-10)
    for v in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, k] += h
            Wm[v, k] -= h
            fd = scale * (oracle.flce_f64(x, Wp, t)[0] - oracle.flce_f64(x, Wm, t)[0]) / (2 * h)
            assert dW[v, k] == pytest.approx(fd, rel=1e-6, abs=1e-10)


def test_flce_grads_equal_chain_rule_through_explicit_logits():
    # dx = dZ W, dW = dZ^T x with dZ the logits gradient of the (separately pinned) CE backward
    T, H, V = 6, 16, 40
    xb = gen.normal_bf16_bits(27, 0, (T, H))
    Wb = gen.normal_bf16_bits(27, 2, (V, H), sigma=0.3)
    t = gen.targets(27, 1, (T,), V)
    widen = lambda b: gen.bf16_bits_to_f32(b).astype(np.float64)  # noqa: E731
    x, W = widen(xb), widen(Wb)
    dz = oracle.ce_grad_f64(x @ W.T, t, None, 1.0 / T)
    dx, dW = oracle.flce_grad_bf16(xb, Wb, t, 1.0)
    np.testing.assert_allclose(dx, dz @ W, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(dW, dz.T @ x, rtol=1e-12, atol=1e-16)
    # rows of dZ sum to zero, so sum_v dW_v = sum_i (sum_v dZ_iv) x_i = 0
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-14)


# ---------------------------------------------------------------- fused linear + JSD backward (student)
@pytest.mark.parametrize("beta,tau,masked", [(0.5, 1.0, False), (0.3, 2.0, True)])
def test_fljsd_student_grads_match_central_differences(beta, tau, masked):
    T, H, V = 3, 4, 6
    xs = gen.normal_f64(28, 0, (T, H))
    Ws = gen.normal_f64(28, 2, (V, H), sigma=0.8)
    xt = gen.normal_f64(28, 3, (T, H))
    Wt = gen.normal_f64(28, 4, (V, H), sigma=0.8)
    keep = np.array([1, 0, 1], np.uint8) if masked else None
    scale = 1.7
    dxs, dWs = oracle.fljsd_grad_f64(xs, Ws, xt, Wt, beta, tau, keep, scale)
    f = lambda a, b: scale * oracle.fljsd_ex_f64(a, b, xt, Wt, beta, tau, keep)[0]  # noqa: E731
    h = 1e-5
    for i in range(T):
        for k in range(H):
            p, m = xs.copy(), xs.copy()
            p[i, k] += h
            m[i, k] -= h
            assert dxs[i, k] == pytest.approx((f(p, Ws) - f(m, Ws)) / (2 * h), rel=1e-6, abs=1e-10)
    for v in range(V):
        for k in range(H):
            p, m = Ws.copy(), Ws.copy()
            p[v, k] += h
            m[v, k] -= h
            assert dWs[v, k] == pytest.approx((f(xs, p) - f(xs, m)) / (2 * h), rel=1e-6, abs=1e-10)
    if masked:
        assert np.all(dxs[1] == 0.0)


def test_fljsd_grads_vanish_at_identical_heads_and_bf16_front_end():
    T, H, V = 4, 8, 20
    x = gen.normal_bf16_bits(29, 0, (T, H))
    W = gen.normal_bf16_bits(29, 2, (V, H), sigma=0.5)
    dxs, dWs = oracle.fljsd_grad_bf16(x, W, x, W)
    assert np.all(np.abs(dxs) < 1e-15) and np.all(np.abs(dWs) < 1e-15)   # JSD minimum: P = Q
    xt = gen.normal_bf16_bits(29, 3, (T, H))
    Wt = gen.normal_bf16_bits(29, 4, (V, H), sigma=0.5)
    widen = lambda b: gen.bf16_bits_to_f32(b).astype(np.float64)  # noqa: E731
    a = oracle.fljsd_grad_bf16(x, W, xt, Wt, 0.4, 1.5, None, 2.0)
    b = oracle.fljsd_grad_f64(widen(x), widen(W), widen(xt), widen(Wt), 0.4, 1.5, None, 2.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fljsd_f64_forward_equals_bf16_oracle_on_widened_inputs():
    T, H, V = 5, 16, 30
    b = [gen.normal_bf16_bits(30, s, shp, sigma=sg) for s, shp, sg in
         ((0, (T, H), 1.0), (2, (V, H), 0.4), (3, (T, H), 1.0), (4, (V, H), 0.4))]
    widen = lambda a: gen.bf16_bits_to_f32(a).astype(np.float64)  # noqa: E731
    keep = np.array([1, 1, 0, 1, 0], np.uint8)
    a = oracle.fljsd_ex_bf16(*b, 0.3, 1.7, keep)
    c = oracle.fljsd_ex_f64(*[widen(x) for x in b], 0.3, 1.7, keep)
    assert a[0] == c[0] and np.array_equal(a[1], c[1])
