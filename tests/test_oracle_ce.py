"""Pins of the cross-entropy oracle against closed forms, invariants and
high-precision brute force (KernelIndex "Cross-entropy loss" and "Vocab-parallel
cross-entropy, Megatron layout", Semantics: per-token loss of a tokens x vocab
logit row against an integer target; flat variant reduced by the mean)."""
import math

import mpmath
import numpy as np
import pytest

import gen
import oracle


def test_single_class_is_zero():
    z = np.array([[3.25], [-7.0], [0.0]])
    m, rows = oracle.ce_f64(z, np.zeros(3, np.int64))
    assert np.all(rows == 0.0) and m == 0.0


@pytest.mark.parametrize("V", [2, 3, 7, 4096, 131072])
@pytest.mark.parametrize("c", [0.0, -3.5, 1e4, -1e4])
def test_equal_logits_give_ln_V(V, c):
    z = np.full((2, V), c)
    m, rows = oracle.ce_f64(z, np.array([0, V - 1]))
    # M + ln(s) - z_t carries a few ulps of |M| of absolute rounding
    tol = 4 * np.spacing(abs(c)) if c else 0.0
    assert rows == pytest.approx([math.log(V)] * 2, rel=1e-14, abs=tol)
    assert m == pytest.approx(math.log(V), rel=1e-14, abs=tol)


@pytest.mark.parametrize("zt,zo", [(0.0, 0.0), (2.0, -1.0), (-30.0, 5.0), (40.0, -40.0)])
def test_two_classes_softplus(zt, zo):
    # loss = ln(1 + e^(z_other - z_target)) for either target position
    want = float(np.logaddexp(0.0, zo - zt))
    _, r0 = oracle.ce_f64(np.array([[zt, zo]]), np.array([0]))
    _, r1 = oracle.ce_f64(np.array([[zo, zt]]), np.array([1]))
    tol = 4 * np.spacing(max(abs(zt), abs(zo)))   # rounding of M + ln(s) - z_t
    assert r0[0] == pytest.approx(want, rel=1e-14, abs=tol)
    assert r1[0] == pytest.approx(want, rel=1e-14, abs=tol)


@pytest.mark.parametrize("L", [0.5, 3.0, 20.0])
def test_one_hot_closed_forms(L):
    V = 50
    z = np.zeros((2, V))
    z[0, 17] = L                 # target holds the spike
    z[1, 3] = L                  # a non-target holds the spike
    m, rows = oracle.ce_f64(z, np.array([17, 40]))
    assert rows[0] == pytest.approx(math.log1p((V - 1) * math.exp(-L)), rel=1e-13)
    assert rows[1] == pytest.approx(math.log(V - 1 + math.exp(L)), rel=1e-13)
    assert m == pytest.approx((rows[0] + rows[1]) / 2, rel=1e-15)


def test_row_shift_invariance():
    z = gen.normal_f64(5, 0, (6, 333), sigma=3.0)
    t = gen.targets(5, 1, (6,), 333)
    _, base = oracle.ce_f64(z, t)
    for c in (1.0, -250.0, 700.0):
        _, shifted = oracle.ce_f64(z + c, t)
        np.testing.assert_allclose(shifted, base, rtol=0, atol=1e-11)


def test_brute_force_probability_route():
    # -ln(e^{z_t} / sum_v e^{z_v}) evaluated at 40 significant digits
    mpmath.mp.dps = 40
    rng = np.random.default_rng(123)
    for V in (2, 3, 4, 5):
        z = np.round(rng.normal(0, 4, size=(3, V)), 3)
        t = rng.integers(0, V, size=3)
        m, rows = oracle.ce_f64(z, t)
        for i in range(3):
            p = mpmath.e ** mpmath.mpf(z[i, t[i]]) / mpmath.fsum(mpmath.e ** mpmath.mpf(v) for v in z[i])
            assert rows[i] == pytest.approx(float(-mpmath.log(p)), rel=1e-14, abs=1e-15)
        assert m == pytest.approx(rows.mean(), rel=1e-15)


def test_integer_logits_hand_values():
    # Row [0, 1, 2] with target 2: ln(1 + e + e^2) - 2 = ln(e^-2 + e^-1 + 1)
    _, r = oracle.ce_f64(np.array([[0.0, 1.0, 2.0]]), np.array([2]))
    assert r[0] == pytest.approx(0.40760596444437567, rel=1e-15)
    # same row, target 0: ln(1 + e + e^2)
    _, r = oracle.ce_f64(np.array([[0.0, 1.0, 2.0]]), np.array([0]))
    assert r[0] == pytest.approx(2.4076059644443806, rel=1e-15)


def test_bad_target_and_nonfinite_give_nan():
    z = np.zeros((4, 8))
    z[2, 5] = np.nan
    z[3, 1] = np.inf
    _, rows = oracle.ce_f64(z, np.array([-1, 8, 0, 0]))
    assert np.all(np.isnan(rows))


def test_f32_front_end_widens_exactly():
    z = gen.normal_f32(0, 0, (7, 129))
    t = gen.targets(0, 1, (7,), 129)
    m32, r32 = oracle.ce_f32(z, t)
    m64, r64 = oracle.ce_f64(z.astype(np.float64), t)
    assert np.array_equal(r32, r64) and m32 == m64


def test_sbv_layout_row_is_s_times_B_plus_b():
    # Each [s, b] row holds one spike of height L = 1 + s*B + b at a
    # non-target position, so its loss is ln(V - 1 + e^L) (closed form).
    S, B, V = 3, 4, 16
    z = np.zeros((S, B, V), np.float32)
    t = np.zeros((S, B), np.int64)
    for s in range(S):
        for b in range(B):
            z[s, b, (s + b) % V] = 1 + s * B + b
            t[s, b] = (s + b + 1) % V
    bits = (z.view(np.uint32) >> 16).astype(np.uint16)   # small integers: exact in bf16
    loss = oracle.ce_sbv_bf16(bits, t)
    for s in range(S):
        for b in range(B):
            L = 1 + s * B + b
            assert loss[s, b] == pytest.approx(math.log(V - 1 + math.exp(L)), rel=1e-14)


def test_statistical_sanity_config_shapes():
    # N(0, sigma^2) logits: E[loss] ~ ln V + sigma^2 / 2 for large V
    z = gen.normal_f32(0, 0, (512, 4096))
    m, _ = oracle.ce_f32(z, gen.targets(0, 1, (512,), 4096))
    assert abs(m - (math.log(4096) + 0.5)) < 0.05
    zb = gen.normal_bf16_bits(0, 0, (64, 4, 4096), sigma=2.0)
    lb = oracle.ce_sbv_bf16(zb, gen.targets(0, 1, (64, 4), 4096))
    assert abs(lb.mean() - (math.log(4096) + 2.0)) < 0.15
