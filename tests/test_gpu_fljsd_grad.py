"""GPU parity of the fused linear + generalized JSD student backward against
the fp64 oracle: dxs = dZs Ws, dWs = dZs^T xs with
dzs = (scale / (n_kept tau)) beta P (ln P - ln M - KL(P || M)).
dZs is rounded to bf16 before the two gradient products: every element is
checked against its own error bound (tests/helpers.py grad_bounds, from the
oracle's exact dZs and g beta P) and the whole gradient normwise within 5e-3,
as for the CE backward.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.helpers import assert_within_bounds, grad_bounds, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def inputs(seed, T, H, V, sw):
    return (gen.normal_bf16_bits(seed, gen.STREAM_X, (T, H)), gen.normal_bf16_bits(seed, gen.STREAM_W, (V, H), sigma=sw),
            gen.normal_bf16_bits(seed, gen.STREAM_XT, (T, H)), gen.normal_bf16_bits(seed, gen.STREAM_WT, (V, H), sigma=sw))


def run(lmho, xs, Ws, xt, Wt, beta=0.5, tau=1.0, keep=None, scale=1.0):
    T, H = xs.shape
    V = Ws.shape[0]
    ws = lmho.workspace(lmho.fljsd_bwd_workspace_bytes(T, H, V))
    loss, dxs, dWs = lmho.fljsd_fwd_bwd_bf16(to_dev_bf16(xs), to_dev_bf16(Ws), to_dev_bf16(xt), to_dev_bf16(Wt), beta, tau,
                                             None if keep is None else to_dev(keep), scale, ws=ws)
    assert lmho.ws_status(ws) == 0
    return (float(loss.item()), lmho.row_losses(ws, T).cpu().numpy().astype(np.float64),
            dxs.cpu().numpy().astype(np.float64), dWs.cpu().numpy().astype(np.float64))


def check(got, ref, bound, what):
    assert_within_bounds(got, ref, bound, what)
    assert np.linalg.norm(got - ref) <= 5e-3 * np.linalg.norm(ref)


CASES = [((5, 64, 37), 0.5, 1.0, False), ((130, 128, 1000), 0.3, 2.0, True), ((64, 256, 4097), 0.5, 1.0, True),
         ((129, 4096, 300), 0.7, 0.8, False), ((256, 512, 2048), 0.5, 1.0, False),
         ((100, 200, 1024), 0.5, 1.0, False)]


@pytest.mark.parametrize("shape,beta,tau,masked", CASES)
def test_fljsd_backward_matches_oracle(gpu_lib, shape, beta, tau, masked):
    T, H, V = shape
    xs, Ws, xt, Wt = inputs(50, T, H, V, sw=2.0 / math.sqrt(H))
    keep = (gen.targets(50, 1, (T,), 4) != 0).astype(np.uint8) if masked else None
    m, rows, dxs, dWs = run(gpu_lib, xs, Ws, xt, Wt, beta, tau, keep, 3.0)
    m_ref, rows_ref = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, beta, tau, keep)
    np.testing.assert_allclose(rows, rows_ref, rtol=1e-3, atol=1e-5)
    assert m == pytest.approx(m_ref, rel=2e-3)
    dz, gbp = oracle.fljsd_dz_bf16(xs, Ws, xt, Wt, beta, tau, keep, 3.0)
    xsd = gen.bf16_bits_to_f32(xs).astype(np.float64)
    Wsd = gen.bf16_bits_to_f32(Ws).astype(np.float64)
    bdx, bdW = grad_bounds(dz, gbp, xsd, Wsd)
    check(dxs, dz @ Wsd, bdx, "dxs")
    check(dWs, dz.T @ xsd, bdW, "dWs")
    if masked:
        assert np.all(dxs[keep == 0] == 0.0)


def test_fljsd_backward_identical_heads_and_loss_matches_forward(gpu_lib):
    T, H, V = 100, 128, 1500
    xs, Ws, xt, Wt = inputs(51, T, H, V, sw=0.2)
    m, rows, dxs, dWs = run(gpu_lib, xs, Ws, xs, Ws)
    assert abs(m) <= 1e-6 and np.abs(dxs).max() <= 1e-6 and np.abs(dWs).max() <= 1e-6
    # the loss of the backward call has the bits of the forward-only call
    m1, r1, _, _ = run(gpu_lib, xs, Ws, xt, Wt, 0.4)
    ws = gpu_lib.workspace(gpu_lib.fljsd_workspace_bytes(T, H, V))
    m2 = float(gpu_lib.fljsd_fwd_bf16(to_dev_bf16(xs), to_dev_bf16(Ws), to_dev_bf16(xt), to_dev_bf16(Wt), 0.4,
                                      ws=ws).item())
    assert m1 == m2 and np.array_equal(r1, gpu_lib.row_losses(ws, T).cpu().numpy().astype(np.float64))


def test_fljsd_backward_full_size_T1024(gpu_lib):
    """Student/teacher [1024, 4096], heads [128256, 4096]: sampled dxs rows
    against the oracle; dWs through <dxs, xs> = <dWs, Ws> and zero column sums."""
    T, H, V = 1024, 4096, 128256
    xs, Ws, xt, Wt = inputs(0, T, H, V, sw=0.02)
    m, rows, dxs, dWs = run(gpu_lib, xs, Ws, xt, Wt)
    idx = sample_rows(T, 3)
    zs = oracle.logits_bf16(xs[idx], Ws)
    zt = oracle.logits_bf16(xt[idx], Wt)
    import scipy.special as sp
    lp = zs - sp.logsumexp(zs, axis=1, keepdims=True)
    lq = zt - sp.logsumexp(zt, axis=1, keepdims=True)
    P, Q = np.exp(lp), np.exp(lq)
    lm = np.log(0.5 * P + 0.5 * Q)
    kl = (P * (lp - lm)).sum(axis=1, keepdims=True)
    dz = (1.0 / T) * 0.5 * P * (lp - lm - kl)
    Wsd = gen.bf16_bits_to_f32(Ws).astype(np.float64)
    xsd = gen.bf16_bits_to_f32(xs).astype(np.float64)
    bdx, _ = grad_bounds(dz, (1.0 / T) * 0.5 * P, xsd[idx], Wsd)
    check(dxs[idx], dz @ Wsd, bdx, "dxs")
    assert float(np.sum(dxs * xsd)) == pytest.approx(float(np.sum(dWs * Wsd)), rel=1e-3)
    assert np.abs(dWs.sum(axis=0)).max() <= 1e-3 * np.abs(dWs).sum(axis=0).max()
    assert np.all(np.isfinite(dWs))
