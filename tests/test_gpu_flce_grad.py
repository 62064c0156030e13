"""GPU parity of the fused linear + cross-entropy backward against the fp64
oracle: dx = dZ W and dW = dZ^T x with dZ = (scale/T)(softmax(x W^T) - onehot).

The kernels round dZ to bf16 before the two gradient products (it is their
tensor-core operand) and accumulate them in fp32: every gradient element is
checked against its own error bound (tests/helpers.py grad_bounds: bf16
rounding and fp32 error of dZ, fp32 accumulation over K, computed from the
oracle's exact dZ), and the whole gradient normwise within 5e-3.  The losses
keep the forward tolerances.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.helpers import assert_within_bounds, ce_error_scale, grad_bounds, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def inputs(seed, T, H, V, sw):
    x = gen.normal_bf16_bits(seed, gen.STREAM_X, (T, H))
    W = gen.normal_bf16_bits(seed, gen.STREAM_W, (V, H), sigma=sw)
    t = gen.targets(seed, gen.STREAM_TARGET, (T,), V)
    return x, W, t


def run(lmho, x, W, t, scale=1.0):
    T, H = x.shape
    V = W.shape[0]
    ws = lmho.workspace(lmho.flce_bwd_workspace_bytes(T, H, V))
    loss, dx, dW = lmho.flce_fwd_bwd_bf16(to_dev_bf16(x), to_dev_bf16(W), to_dev(t), scale, ws=ws)
    assert lmho.ws_status(ws) == 0
    return (float(loss.item()), lmho.row_losses(ws, T).cpu().numpy().astype(np.float64),
            dx.cpu().numpy().astype(np.float64), dW.cpu().numpy().astype(np.float64))


def check_grads(x, W, t, scale, dx, dW, rows=None):
    """dx (all rows, or the given token rows of it) and dW (unless None)
    against the oracle's dZ products, every element within its own bound."""
    T = x.shape[0]
    sel = np.arange(T) if rows is None else np.asarray(rows)
    dz = oracle.ce_grad_f64(oracle.logits_bf16(x[sel], W), t[sel], None, scale / T)
    S = ce_error_scale(dz, t[sel], scale / T)
    xd = gen.bf16_bits_to_f32(x[sel]).astype(np.float64)
    Wd = gen.bf16_bits_to_f32(W).astype(np.float64)
    bdx, bdW = grad_bounds(dz, S, xd, Wd)
    dx_ref = dz @ Wd
    assert_within_bounds(dx[sel], dx_ref, bdx, "dx")
    assert np.linalg.norm(dx[sel] - dx_ref) <= 5e-3 * np.linalg.norm(dx_ref)
    if dW is not None:
        dW_ref = dz.T @ xd
        assert_within_bounds(dW, dW_ref, bdW, "dW")
        assert np.linalg.norm(dW - dW_ref) <= 5e-3 * np.linalg.norm(dW_ref)


SHAPES = [(1, 64, 1), (5, 64, 37), (130, 128, 1000), (257, 200, 4097), (64, 1024, 513), (256, 512, 4096),
          (70, 8, 300), (129, 16, 2049),   # H = 8, 16: MN-major boxes mostly past the edge (zero fill)
          (300, 200, 1024), (33, 72, 640)]  # V whole 64-wide chunks, H not: 3-D map for dZ, 2-D for W and x


@pytest.mark.parametrize("T,H,V", SHAPES)
def test_flce_backward_matches_oracle(gpu_lib, T, H, V):
    x, W, t = inputs(40, T, H, V, sw=2.0 / math.sqrt(H))
    m, rows, dx, dW = run(gpu_lib, x, W, t, 2.0)
    m_ref, rows_ref = oracle.flce_bf16(x, W, t)
    np.testing.assert_allclose(rows, rows_ref, rtol=1e-4, atol=1e-5)
    assert m == pytest.approx(m_ref, rel=2e-3)
    if V == 1:  # softmax of one class is 1: every gradient is exactly 0
        assert np.all(dx == 0) and np.all(dW == 0)
        return
    check_grads(x, W, t, 2.0, dx, dW)


def test_flce_backward_bad_target_and_determinism(gpu_lib):
    T, H, V = 40, 128, 700
    x, W, t = inputs(41, T, H, V, sw=0.2)
    a = run(gpu_lib, x, W, t)
    b = run(gpu_lib, x, W, t)
    assert a[0] == b[0] and np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])
    t[7] = V
    m, rows, dx, dW = run(gpu_lib, x, W, t)
    assert math.isnan(m) and np.isnan(rows[7]) and np.all(np.isnan(dx[7])) and np.all(np.isnan(dW))
    assert np.all(np.isfinite(np.delete(dx, 7, axis=0)))


def test_flce_backward_full_size_batch2(gpu_lib):
    """x [2048, 4096], W [128256, 4096] bf16: sampled dx rows against the
    oracle; dW through identities that hold at any size:
    <dx, x> = <dW, W> (both equal sum dZ * Z) and sum_v dW_v = 0."""
    T, H, V = 2048, 4096, 128256
    x, W, t = inputs(0, T, H, V, sw=0.02)
    m, rows, dx, dW = run(gpu_lib, x, W, t)
    idx = sample_rows(T, 6)
    xs = gen.bf16_bits_to_f32(x).astype(np.float64)
    Ws = gen.bf16_bits_to_f32(W).astype(np.float64)
    check_grads(x, W, t, 1.0, dx, None, rows=idx)
    lhs = float(np.sum(dx * xs))
    rhs = float(np.sum(dW * Ws))
    assert lhs == pytest.approx(rhs, rel=1e-3)
    colsum = np.abs(dW.sum(axis=0)).max()
    assert colsum <= 1e-3 * np.abs(dW).sum(axis=0).max()
    assert np.all(np.isfinite(dW))


def test_flce_backward_split_k_is_bitwise_reproducible(gpu_lib):
    """dx with too few output tiles to fill the GPU is cut along K (here 65
    k-blocks into slices of 17, 17, 17 and 14) and the fp32 slices are summed
    in slice order: repeated calls give the same bits, and the result matches
    the oracle."""
    T, H, V = 257, 200, 4097
    x, W, t = inputs(42, T, H, V, sw=0.1)
    a = run(gpu_lib, x, W, t)
    b = run(gpu_lib, x, W, t)
    assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])
    check_grads(x, W, t, 1.0, a[2], a[3])
