"""Pins of the fused-linear oracles (KernelIndex "Fused linear + CPO loss":
x [batch, seq, hidden], weight [vocab, hidden], integer targets, loss [1],
computed without materialising logits; "Fused linear + JSD": student and
teacher activations through separate vocab x hidden heads, generalized JSD with
beta 0.5, batchmean)."""
import math

import numpy as np
import pytest
import scipy.special as sp

import gen
import oracle


def bits(a):
    """Round float32 values to bf16 bit patterns (nearest even)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def widen(b):
    return gen.bf16_bits_to_f32(b).astype(np.float64)


def small_case(T=5, H=24, V=37, seed=3):
    x = gen.normal_bf16_bits(seed, 0, (T, H))
    W = gen.normal_bf16_bits(seed, 2, (V, H), sigma=0.5)
    t = gen.targets(seed, 1, (T,), V)
    return x, W, t


# ---------------------------------------------------------------- fused CE

def test_logits_are_x_times_W_transpose():
    x, W, _ = small_case()
    z = oracle.logits_bf16(x, W)
    assert z.shape == (5, 37)
    np.testing.assert_allclose(z, widen(x) @ widen(W).T, rtol=1e-13, atol=1e-13)


def test_flce_equals_ce_of_explicit_logits():
    x, W, t = small_case()
    m, rows = oracle.flce_bf16(x, W, t, threads=2)
    m_ref, rows_ref = oracle.ce_f64(widen(x) @ widen(W).T, t)
    np.testing.assert_allclose(rows, rows_ref, rtol=1e-12)
    assert m == pytest.approx(m_ref, rel=1e-12)


@pytest.mark.parametrize("V", [1, 2, 37, 1000])
def test_flce_zero_input_gives_ln_V(V):
    x = np.zeros((3, 16), np.uint16)
    W = gen.normal_bf16_bits(0, 2, (V, 16))
    m, rows = oracle.flce_bf16(x, W, gen.targets(0, 1, (3,), V))
    assert np.all(rows == pytest.approx(math.log(V), rel=1e-15, abs=1e-300))


def test_flce_identical_head_rows_give_ln_V():
    V, H = 64, 40
    row = gen.normal_bf16_bits(1, 2, (1, H))
    W = np.repeat(row, V, axis=0)
    x = gen.normal_bf16_bits(1, 0, (4, H))
    _, rows = oracle.flce_bf16(x, W, gen.targets(1, 1, (4,), V))
    np.testing.assert_allclose(rows, math.log(V), rtol=1e-14)


def test_flce_threads_do_not_change_bits():
    x, W, t = small_case(T=9)
    a = oracle.flce_bf16(x, W, t, threads=1)
    b = oracle.flce_bf16(x, W, t, threads=4)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


def test_flce_target_picks_the_right_column():
    # x = e_0, W[v, 0] = v/8 (exact in bf16): z_v = v/8, so the loss of target t
    # is ln(sum_v e^{v/8}) - t/8, a closed form of the geometric series.
    V, H = 33, 8
    x = np.zeros((V, H), np.float32)
    x[:, 0] = 1.0
    W = np.zeros((V, H), np.float32)
    W[:, 0] = np.arange(V) / 8.0
    t = np.arange(V, dtype=np.int64)
    _, rows = oracle.flce_bf16(bits(x), bits(W), t)
    q = math.exp(1 / 8)
    lse = math.log((q ** V - 1) / (q - 1))
    np.testing.assert_allclose(rows, lse - t / 8.0, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- JSD

def entropy(p):
    return -sp.xlogy(p, p).sum(axis=-1)


@pytest.mark.parametrize("beta", [0.5, 0.2, 0.9])
def test_jsd_entropy_identity(beta):
    # JSD_beta = H(M) - beta H(P) - (1 - beta) H(Q)  (Shannon entropies)
    zs = gen.normal_f64(7, 0, (6, 50), sigma=2.0)
    zt = gen.normal_f64(7, 3, (6, 50), sigma=2.0)
    m, rows = oracle.jsd_f64(zs, zt, beta)
    P, Q = sp.softmax(zs, axis=1), sp.softmax(zt, axis=1)
    want = entropy(beta * P + (1 - beta) * Q) - beta * entropy(P) - (1 - beta) * entropy(Q)
    np.testing.assert_allclose(rows, want, rtol=1e-12, atol=1e-15)
    assert m == pytest.approx(want.mean(), rel=1e-12)


def test_jsd_identical_is_zero_and_bounded():
    z = gen.normal_f64(8, 0, (5, 300), sigma=3.0)
    _, rows = oracle.jsd_f64(z, z, 0.5)
    assert np.all(np.abs(rows) < 1e-14)
    zt = gen.normal_f64(8, 3, (5, 300), sigma=3.0)
    _, rows = oracle.jsd_f64(z, zt, 0.5)
    assert np.all(rows >= 0) and np.all(rows <= math.log(2))


@pytest.mark.parametrize("beta", [0.5, 0.25])
def test_jsd_disjoint_supports_is_binary_entropy(beta):
    zs = np.array([[30.0, 30.0, -30.0, -30.0]])
    zt = np.array([[-30.0, -30.0, 30.0, 30.0]])
    _, rows = oracle.jsd_f64(zs, zt, beta)
    hb = -beta * math.log(beta) - (1 - beta) * math.log(1 - beta)
    assert rows[0] == pytest.approx(hb, rel=1e-12)


def test_jsd_symmetry_and_beta_swap():
    zs = gen.normal_f64(9, 0, (4, 64))
    zt = gen.normal_f64(9, 3, (4, 64))
    a = oracle.jsd_f64(zs, zt, 0.5)[1]
    b = oracle.jsd_f64(zt, zs, 0.5)[1]
    np.testing.assert_allclose(a, b, rtol=1e-13)
    c = oracle.jsd_f64(zs, zt, 0.3)[1]
    d = oracle.jsd_f64(zt, zs, 0.7)[1]
    np.testing.assert_allclose(c, d, rtol=1e-13)


def test_jsd_orientation_student_is_P():
    # For small beta, JSD_beta / beta -> KL(P || Q) with P the first (student) argument.
    zs = gen.normal_f64(10, 0, (3, 20), sigma=1.5)
    zt = gen.normal_f64(10, 3, (3, 20), sigma=1.5)
    beta = 1e-7
    _, rows = oracle.jsd_f64(zs, zt, beta)
    P, Q = sp.softmax(zs, axis=1), sp.softmax(zt, axis=1)
    kl_pq = sp.rel_entr(P, Q).sum(axis=1)
    kl_qp = sp.rel_entr(Q, P).sum(axis=1)
    np.testing.assert_allclose(rows / beta, kl_pq, rtol=1e-4)
    assert np.all(np.abs(kl_pq - kl_qp) > 1e-2)


def test_fljsd_equals_jsd_of_explicit_logits():
    T, H, V = 4, 32, 45
    xs = gen.normal_bf16_bits(11, 0, (T, H))
    Ws = gen.normal_bf16_bits(11, 2, (V, H), sigma=0.4)
    xt = gen.normal_bf16_bits(11, 3, (T, H))
    Wt = gen.normal_bf16_bits(11, 4, (V, H), sigma=0.4)
    for beta in (0.5, 0.3):
        m, rows = oracle.fljsd_bf16(xs, Ws, xt, Wt, beta, threads=3)
        m_ref, rows_ref = oracle.jsd_f64(widen(xs) @ widen(Ws).T, widen(xt) @ widen(Wt).T, beta)
        np.testing.assert_allclose(rows, rows_ref, rtol=1e-12, atol=1e-15)
        assert m == pytest.approx(m_ref, rel=1e-12)


def test_fljsd_same_student_and_teacher_is_zero():
    T, H, V = 3, 16, 70
    x = gen.normal_bf16_bits(12, 0, (T, H))
    W = gen.normal_bf16_bits(12, 2, (V, H))
    m, rows = oracle.fljsd_bf16(x, W, x, W, 0.5)
    assert abs(m) < 1e-14 and np.all(np.abs(rows) < 1e-14)


# ---------------------------------------------------------------- JSD variant (temperature, mask)

def _jsd_case(seed=15, T=6, H=32, V=57, sw=0.5):
    return (gen.normal_bf16_bits(seed, 0, (T, H)), gen.normal_bf16_bits(seed, 2, (V, H), sigma=sw),
            gen.normal_bf16_bits(seed, 3, (T, H)), gen.normal_bf16_bits(seed, 4, (V, H), sigma=sw))


def test_jsd_ex_defaults_equal_base():
    xs, Ws, xt, Wt = _jsd_case()
    a = oracle.fljsd_bf16(xs, Ws, xt, Wt, 0.3)
    b = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, 0.3, 1.0, None)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


def test_jsd_ex_temperature_two_equals_halved_inputs():
    # tau = 2 divides every logit by 2; so does halving x (exact in bf16: an exponent step)
    xs, Ws, xt, Wt = _jsd_case()
    half = lambda b: bits(widen(b).astype(np.float32) / 2)  # noqa: E731
    m2, r2 = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, 0.5, 2.0)
    mh, rh = oracle.fljsd_bf16(half(xs), Ws, half(xt), Wt, 0.5)
    np.testing.assert_allclose(r2, rh, rtol=1e-12, atol=1e-16)
    assert m2 == pytest.approx(mh, rel=1e-12)


def test_jsd_ex_high_temperature_goes_to_zero():
    # tau -> infinity flattens both distributions to uniform: JSD -> 0 like 1/tau^2
    xs, Ws, xt, Wt = _jsd_case()
    m1, _ = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, 0.5, 1e3)
    m2, _ = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, 0.5, 2e3)
    assert 0 < m2 < m1 < 1e-5
    assert m1 / m2 == pytest.approx(4.0, rel=1e-2)


def test_jsd_ex_mask_means_over_kept_tokens():
    xs, Ws, xt, Wt = _jsd_case()
    keep = np.array([1, 0, 1, 1, 0, 1], np.uint8)
    _, base = oracle.fljsd_bf16(xs, Ws, xt, Wt, 0.5)
    m, rows = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, 0.5, 1.0, keep)
    assert np.all(rows[keep == 0] == 0.0)
    np.testing.assert_array_equal(rows[keep == 1], base[keep == 1])
    assert m == pytest.approx(base[keep == 1].mean(), rel=1e-15)
    m0, rows0 = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, 0.5, 1.0, np.zeros(6, np.uint8))
    assert m0 == 0.0 and np.all(rows0 == 0.0)
