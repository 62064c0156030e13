"""GPU parity of the fused linear + CPO loss (page "Fused linear + CPO loss";
the objective is the published CPO, chosen = first half of the batch) against
the fp64 oracle.

Tolerances: per-token CE losses as the fused CE (relative 1e-4, absolute
1e-5); a sequence log-likelihood sums S of them, so |d lp| <= 1e-4 * sum |l|
+ 1e-5 S; the loss scalar relative 2e-3 (the fused-linear scalar tolerance).
Gradients as the fused CE backward (dZ is a bf16 operand): every element
within its own error bound (tests/helpers.py grad_bounds, from the oracle's
exact dZ = scale w_i (softmax - onehot) with the oracle's row weights w_i),
normwise within 5e-3.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.helpers import assert_within_bounds, ce_error_scale, grad_bounds, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def inputs(seed, B, S, H, V, sw):
    x = gen.normal_bf16_bits(seed, gen.STREAM_X, (B, S, H))
    W = gen.normal_bf16_bits(seed, gen.STREAM_W, (V, H), sigma=sw)
    t = gen.targets(seed, gen.STREAM_TARGET, (B, S), V)
    return x, W, t


def check_lp(lp, lp_ref, rows_ref):
    S = rows_ref.shape[1]
    tol = 1e-4 * np.abs(rows_ref).sum(axis=1) + 1e-5 * S
    assert np.all(np.abs(lp - lp_ref) <= tol), (lp, lp_ref)


def check_grads(xf, W, tf, w_rows, scale, dx, dW, rows=None):
    """dx (all rows, or the given token rows) and dW (unless None) against the
    oracle's dZ products; w_rows = the oracle's d loss / d l_i of every token."""
    sel = np.arange(xf.shape[0]) if rows is None else np.asarray(rows)
    dz = oracle.ce_grad_f64(oracle.logits_bf16(xf[sel], W), tf[sel], w_rows[sel], scale)
    S = ce_error_scale(dz, tf[sel], scale * w_rows[sel])
    xd = gen.bf16_bits_to_f32(xf[sel]).astype(np.float64)
    Wd = gen.bf16_bits_to_f32(W).astype(np.float64)
    bdx, bdW = grad_bounds(dz, S, xd, Wd)
    dx_ref = dz @ Wd
    assert_within_bounds(dx[sel], dx_ref, bdx, "dx")
    assert np.linalg.norm(dx[sel] - dx_ref) <= 5e-3 * np.linalg.norm(dx_ref)
    if dW is not None:
        dW_ref = dz.T @ xd
        assert_within_bounds(dW, dW_ref, bdW, "dW")
        assert np.linalg.norm(dW - dW_ref) <= 5e-3 * np.linalg.norm(dW_ref)


SHAPES = [(2, 1, 64, 37), (2, 3, 64, 513), (4, 33, 128, 1000), (6, 50, 200, 4097), (2, 130, 256, 4096),
          (8, 16, 512, 2048)]


@pytest.mark.parametrize("B,S,H,V", SHAPES)
def test_cpo_forward_matches_oracle(gpu_lib, B, S, H, V):
    x, W, t = inputs(50, B, S, H, V, sw=2.0 / math.sqrt(H))
    beta, alpha = 0.7, 1.3
    ws = gpu_lib.workspace(gpu_lib.flce_cpo_workspace_bytes(B, S, H, V))
    loss, lp = gpu_lib.flce_cpo_fwd_bf16(to_dev_bf16(x), to_dev_bf16(W), to_dev(t), beta, alpha, ws=ws)
    assert gpu_lib.ws_status(ws) == 0
    m_ref, rows_ref, lp_ref = oracle.cpo_bf16(x, W, t, beta, alpha)
    rows = gpu_lib.row_losses(ws, B * S).cpu().numpy().astype(np.float64).reshape(B, S)
    np.testing.assert_allclose(rows, rows_ref, rtol=1e-4, atol=1e-5)
    check_lp(lp.cpu().numpy().astype(np.float64), lp_ref, rows_ref)
    assert float(loss.item()) == pytest.approx(m_ref, rel=2e-3)


@pytest.mark.parametrize("B,S,H,V", SHAPES)
def test_cpo_backward_matches_oracle(gpu_lib, B, S, H, V):
    x, W, t = inputs(51, B, S, H, V, sw=2.0 / math.sqrt(H))
    beta, alpha, scale = 0.5, 1.0, 3.0
    ws = gpu_lib.workspace(gpu_lib.flce_cpo_bwd_workspace_bytes(B, S, H, V))
    loss, lp, dx, dW = gpu_lib.flce_cpo_fwd_bwd_bf16(to_dev_bf16(x), to_dev_bf16(W), to_dev(t), beta, alpha, scale,
                                                     ws=ws)
    assert gpu_lib.ws_status(ws) == 0
    m_ref, rows_ref, lp_ref = oracle.cpo_bf16(x, W, t, beta, alpha)
    assert float(loss.item()) == pytest.approx(m_ref, rel=2e-3)
    check_lp(lp.cpu().numpy().astype(np.float64), lp_ref, rows_ref)
    if V == 1:
        return
    T = B * S
    _, _, w_rows = oracle.cpo_combine(rows_ref, beta, alpha)
    check_grads(x.reshape(T, H), W, t.reshape(T), np.asarray(w_rows).reshape(T), scale,
                dx.cpu().numpy().astype(np.float64).reshape(T, H), dW.cpu().numpy().astype(np.float64))
    # the row weights are the oracle gradient's: its dx is the same dZ product
    dx_ref, _ = oracle.cpo_grad_bf16(x, W, t, beta, alpha, scale)
    dz = oracle.ce_grad_f64(oracle.logits_bf16(x.reshape(T, H), W), t.reshape(T), np.asarray(w_rows).reshape(T), scale)
    np.testing.assert_allclose(dx_ref.reshape(T, H), dz @ gen.bf16_bits_to_f32(W).astype(np.float64),
                               rtol=1e-9, atol=1e-15)


def test_cpo_identical_answers_and_alpha_zero(gpu_lib):
    # rejected = chosen: every margin is exactly 0 on the GPU too (same bits in,
    # same fixed-order sums), so with alpha = 0 the loss is ln 2 to fp32 rounding
    B, S, H, V = 4, 40, 256, 3000
    x, W, t = inputs(52, B, S, H, V, sw=0.1)
    x[2:] = x[:2]
    t[2:] = t[:2]
    loss, lp = gpu_lib.flce_cpo_fwd_bf16(to_dev_bf16(x), to_dev_bf16(W), to_dev(t), 0.1, 0.0)
    lp = lp.cpu().numpy()
    assert np.array_equal(lp[:2], lp[2:])
    assert float(loss.item()) == pytest.approx(math.log(2), rel=1e-6)


def test_cpo_bad_target_determinism_and_errors(gpu_lib):
    B, S, H, V = 4, 20, 128, 700
    x, W, t = inputs(53, B, S, H, V, sw=0.2)
    run = lambda tt: gpu_lib.flce_cpo_fwd_bwd_bf16(to_dev_bf16(x), to_dev_bf16(W), to_dev(tt), 0.1, 1.0)  # noqa: E731
    a = [r.cpu() for r in run(t)]
    b = [r.cpu() for r in run(t)]
    assert all(torch.equal(p, q) for p, q in zip(a, b))
    t2 = t.copy()
    t2[3, 5] = V          # rejected sequence 3 = pair 1
    loss, lp, dx, dW = [r.cpu().numpy() for r in run(t2)]
    assert math.isnan(loss[0]) and np.isnan(lp[3]) and np.all(np.isfinite(lp[:3]))
    assert np.all(np.isnan(dx[1])) and np.all(np.isnan(dx[3])) and np.all(np.isnan(dW))
    assert np.all(np.isfinite(dx[0])) and np.all(np.isfinite(dx[2]))
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    with pytest.raises(gpu_lib.LmhoError) as e:
        gpu_lib.flce_cpo_fwd_bf16(xd[:3], Wd, td[:3])            # odd batch
    assert e.value.status == gpu_lib.LMHO_ERR_INVALID_ARG
    with pytest.raises(gpu_lib.LmhoError) as e:
        gpu_lib.flce_cpo_fwd_bf16(xd, Wd, td, beta=0.0)
    assert e.value.status == gpu_lib.LMHO_ERR_INVALID_ARG


def test_cpo_full_size_batch2(gpu_lib):
    """x [2, 1024, 4096], W [128256, 4096] bf16 (the page's batch-2 workload):
    sampled per-token losses against the oracle; the pair combination of the
    kernel's own per-token losses against the oracle's combination; sampled dx
    rows through the oracle's row weights; dW through <dx, x> = <dW, W> and
    zero column sums."""
    B, S, H, V = 2, 1024, 4096, 128256
    x, W, t = inputs(0, B, S, H, V, sw=0.02)
    T = B * S
    ws = gpu_lib.workspace(gpu_lib.flce_cpo_bwd_workspace_bytes(B, S, H, V))
    loss, lp, dx, dW = gpu_lib.flce_cpo_fwd_bwd_bf16(to_dev_bf16(x), to_dev_bf16(W), to_dev(t), 0.1, 1.0, ws=ws)
    assert gpu_lib.ws_status(ws) == 0
    rows = gpu_lib.row_losses(ws, T).cpu().numpy().astype(np.float64)
    idx = sample_rows(T, 6)
    xf, tf = x.reshape(T, H), t.reshape(T)
    _, rows_ref = oracle.flce_bf16(xf[idx], W, tf[idx])
    np.testing.assert_allclose(rows[idx], rows_ref, rtol=1e-4, atol=1e-5)
    m_c, lp_c, w_c = oracle.cpo_combine(rows.reshape(B, S), 0.1, 1.0)
    assert float(loss.item()) == pytest.approx(m_c, rel=2e-3)
    check_lp(lp.cpu().numpy().astype(np.float64), lp_c, rows.reshape(B, S))
    Ws = gen.bf16_bits_to_f32(W).astype(np.float64)
    dxn = dx.cpu().numpy().astype(np.float64).reshape(T, H)
    check_grads(xf, W, tf, np.asarray(w_c).reshape(T), 1.0, dxn, None, rows=idx)
    dWn = dW.cpu().numpy().astype(np.float64)
    xs = gen.bf16_bits_to_f32(xf).astype(np.float64)
    assert float(np.sum(dxn * xs)) == pytest.approx(float(np.sum(dWn * Ws)), rel=1e-3)
    assert np.abs(dWn.sum(axis=0)).max() <= 1e-3 * np.abs(dWn).sum(axis=0).max()


def test_cpo_workspace_reuse_leaves_ticket_at_zero(gpu_lib):
    """Both finalisers of a CPO call (the CE mean and the pair combination) use
    the workspace's ticket word and must leave it at zero: repeated calls on one
    workspace, forward and forward + backward, give identical bits."""
    B, S, H, V = 4, 40, 128, 900
    x, W, t = inputs(54, B, S, H, V, sw=0.2)
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    ws = gpu_lib.workspace(gpu_lib.flce_cpo_bwd_workspace_bytes(B, S, H, V))
    outs = [gpu_lib.flce_cpo_fwd_bwd_bf16(xd, Wd, td, 0.3, 1.0, ws=ws) for _ in range(3)]
    outs = [[o.clone() for o in r] for r in outs]
    assert int(ws[-256:].view(torch.int32)[1].item()) == 0
    for r in outs[1:]:
        assert all(torch.equal(p, q) for p, q in zip(r, outs[0]))
    f = [gpu_lib.flce_cpo_fwd_bf16(xd, Wd, td, 0.3, 1.0, ws=ws)[0].clone() for _ in range(2)]
    assert torch.equal(f[0], f[1]) and torch.equal(f[0], outs[0][0])
    assert int(ws[-256:].view(torch.int32)[1].item()) == 0
