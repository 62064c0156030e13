"""Pins of the per-element error bounds the fused-backward parity tests use
(tests/helpers.py: grad_bounds).  The kernels round dZ to bf16 and
accumulate the gradient products in fp32; here that arithmetic is done by hand
on the host from the oracle's exact dZ: dZ perturbed within its fp32 error
model, rounded to bf16 (round to nearest even), and the products accumulated
in fp32 sixteen terms at a time.  Every element of the result must stay
inside its own bound, for the cross-entropy, the JSD and the CPO gradients;
a planted mistake (a dropped target term) must not."""
import math

import numpy as np
import pytest

import gen
import oracle
from tests.helpers import DZ_ERR, assert_within_bounds, ce_error_scale, grad_bounds


def rne_bf16(a):
    """fp64 -> nearest-even bf16 value (through fp32, as the kernel's
    cvt.rn.bf16x2.f32 sees an fp32 operand), returned as fp64."""
    f = np.asarray(a, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


def f32_accumulate(A, B):
    """A [M, K] @ B [K, N] with an fp32 accumulator advanced 16 products at a
    time (each group's sum exact, then rounded into the fp32 total)."""
    M, K = A.shape
    acc = np.zeros((M, B.shape[1]), np.float32)
    for k0 in range(0, K, 16):
        acc = (acc.astype(np.float64) + A[:, k0:k0 + 16] @ B[k0:k0 + 16]).astype(np.float32)
    return acc.astype(np.float64)


def kernel_emulation(dz, S, x, W, seed):
    rng = np.random.default_rng(seed)
    dz_gpu = dz + 0.5 * DZ_ERR * S * rng.uniform(-1, 1, dz.shape)
    q = rne_bf16(dz_gpu)
    return f32_accumulate(q, W), f32_accumulate(q.T, x)


def bf16_vals(bits):
    return gen.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("T,H,V", [(7, 16, 40), (33, 64, 300), (64, 32, 1025)])
def test_flce_bound_holds_for_bf16_rounded_dz(T, H, V):
    x = gen.normal_bf16_bits(60, 0, (T, H))
    W = gen.normal_bf16_bits(60, 2, (V, H), sigma=2.0 / math.sqrt(H))
    t = gen.targets(60, 1, (T,), V)
    scale = 3.0
    dz = oracle.ce_grad_f64(oracle.logits_bf16(x, W), t, None, scale / T)
    S = ce_error_scale(dz, t, scale / T)
    xd, Wd = bf16_vals(x), bf16_vals(W)
    dx_ref, dW_ref = oracle.flce_grad_bf16(x, W, t, scale)
    bdx, bdW = grad_bounds(dz, S, xd, Wd)
    for seed in range(3):
        dx, dW = kernel_emulation(dz, S, xd, Wd, seed)
        assert_within_bounds(dx, dx_ref, bdx, "dx")
        assert_within_bounds(dW, dW_ref, bdW, "dW")
    # the bound is not vacuous: a dropped target term breaks it
    dz_bad = dz.copy()
    dz_bad[np.arange(T), t] = 0.0
    dx_bad, _ = kernel_emulation(dz_bad, S, xd, Wd, 9)
    with pytest.raises(AssertionError):
        assert_within_bounds(dx_bad, dx_ref, bdx, "dx")


@pytest.mark.parametrize("beta,tau,masked", [(0.5, 1.0, False), (0.3, 2.0, True)])
def test_fljsd_bound_holds_for_bf16_rounded_dz(beta, tau, masked):
    T, H, V = 24, 32, 500
    xs = gen.normal_bf16_bits(61, 0, (T, H))
    Ws = gen.normal_bf16_bits(61, 2, (V, H), sigma=2.0 / math.sqrt(H))
    xt = gen.normal_bf16_bits(61, 3, (T, H))
    Wt = gen.normal_bf16_bits(61, 4, (V, H), sigma=2.0 / math.sqrt(H))
    keep = (gen.targets(61, 1, (T,), 4) != 0).astype(np.uint8) if masked else None
    dz, gbp = oracle.fljsd_dz_bf16(xs, Ws, xt, Wt, beta, tau, keep, 2.0)
    dx_ref, dW_ref = oracle.fljsd_grad_bf16(xs, Ws, xt, Wt, beta, tau, keep, 2.0)
    # the oracle's dZs is the one its gradient multiplies
    np.testing.assert_allclose(dz @ bf16_vals(Ws), dx_ref, rtol=1e-12, atol=1e-15)
    bdx, bdW = grad_bounds(dz, gbp, bf16_vals(xs), bf16_vals(Ws))
    for seed in range(3):
        dx, dW = kernel_emulation(dz, gbp, bf16_vals(xs), bf16_vals(Ws), seed)
        assert_within_bounds(dx, dx_ref, bdx, "dxs")
        assert_within_bounds(dW, dW_ref, bdW, "dWs")


def test_cpo_bound_holds_for_bf16_rounded_dz():
    B, S_, H, V = 4, 6, 32, 200
    T = B * S_
    x = gen.normal_bf16_bits(62, 0, (T, H))
    W = gen.normal_bf16_bits(62, 2, (V, H), sigma=2.0 / math.sqrt(H))
    t = gen.targets(62, 1, (T,), V)
    _, rows = oracle.flce_bf16(x, W, t)
    _, _, row_w = oracle.cpo_combine(rows.reshape(B, S_), 0.1, 1.0)
    row_w = row_w.reshape(T)
    dz = oracle.ce_grad_f64(oracle.logits_bf16(x, W), t, row_w, 1.5)
    S = ce_error_scale(dz, t, 1.5 * row_w)
    dx_ref, dW_ref = oracle.cpo_grad_bf16(x.reshape(B, S_, H), W, t.reshape(B, S_), 0.1, 1.0, 1.5)
    xd, Wd = bf16_vals(x), bf16_vals(W)
    bdx, bdW = grad_bounds(dz, S, xd, Wd)
    dx, dW = kernel_emulation(dz, S, xd, Wd, 0)
    assert_within_bounds(dx, dx_ref.reshape(T, H), bdx, "dx")
    assert_within_bounds(dW, dW_ref, bdW, "dW")
