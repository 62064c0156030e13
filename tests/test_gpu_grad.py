"""GPU parity of the cross-entropy forward + backward (loss and gradient with
respect to the logits in one pass) against the fp64 oracle.

Losses: the forward tolerances (fp32 relative 1e-5; bf16 logits 2e-3
absolute per token).  Gradients: fp32 relative 2e-5 plus 1e-7 * g absolute
(ex2.approx and the fp32 log-sum-exp leave ~1e-6 relative on softmax); bf16
gradients are rounded to nearest even, so relative 4.5e-3 (half a bf16 ulp is
2^-8 = 3.9e-3 relative) plus the same absolute floor.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.helpers import sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def bf16_to_f64(t):
    return (t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_flat(lmho, z, t, scale, dlogits=None):
    T, V = z.shape
    ws = lmho.workspace(lmho.ce_workspace_bytes(T, V))
    loss, dz = lmho.ce_fwd_bwd_f32(to_dev(z), to_dev(t), scale, ws=ws, dlogits=dlogits)
    torch.cuda.synchronize()
    return float(loss.item()), lmho.row_losses(ws, T).cpu().numpy().astype(np.float64), dz


FLAT = [(1, 1), (3, 5), (4, 8), (7, 4095), (33, 4097), (64, 4096), (300, 1000), (5, 16385), (3, 65537),
        (2, 131071), (2, 200001), (9000, 1024), (3, 30000), (2, 32768), (2, 24577)]


@pytest.mark.parametrize("T,V", FLAT)
def test_flat_fwd_bwd_matches_oracle(gpu_lib, T, V):
    z = gen.normal_f32(30, 0, (T, V))
    t = gen.targets(30, 1, (T,), V)
    scale = 1.7
    m, rows, dz = run_flat(gpu_lib, z, t, scale)
    m_ref, rows_ref = oracle.ce_f32(z, t)
    np.testing.assert_allclose(rows, rows_ref, rtol=1e-5, atol=1e-6)
    assert m == pytest.approx(m_ref, rel=1e-5, abs=1e-6)
    ref = oracle.ce_grad_f32(z, t, scale)
    g = scale / T
    np.testing.assert_allclose(dz.cpu().numpy(), ref, rtol=2e-5, atol=1e-7 * g)


def test_flat_gradient_buffer_with_other_alignment(gpu_lib):
    # dlogits rows 4 bytes off the logits' 16-byte phase: the scalar store path
    T, V = 37, 1024
    z = gen.normal_f32(31, 0, (T, V))
    t = gen.targets(31, 1, (T,), V)
    big = torch.empty(T * V + 1, dtype=torch.float32, device="cuda")
    dz = big[1:].view(T, V)
    _, _, out = run_flat(gpu_lib, z, t, 1.0, dlogits=dz)
    np.testing.assert_allclose(out.cpu().numpy(), oracle.ce_grad_f32(z, t, 1.0), rtol=2e-5, atol=1e-7 / T)


def test_flat_bad_target_rows_are_nan_and_sums_vanish(gpu_lib):
    T, V = 6, 3000
    z = gen.normal_f32(32, 0, (T, V))
    t = gen.targets(32, 1, (T,), V)
    t[1] = -3
    m, rows, dz = run_flat(gpu_lib, z, t, 1.0)
    d = dz.cpu().numpy().astype(np.float64)
    assert np.isnan(rows[1]) and math.isnan(m) and np.all(np.isnan(d[1]))
    keep = [0, 2, 3, 4, 5]
    assert np.all(np.isfinite(d[keep]))
    np.testing.assert_allclose(d[keep].sum(axis=1), 0.0, atol=1e-6 / T)


def test_flat_fwd_bwd_deterministic(gpu_lib):
    T, V = 500, 20000
    z = to_dev(gen.normal_f32(33, 0, (T, V)))
    t = to_dev(gen.targets(33, 1, (T,), V))
    ws = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(T, V))
    a = [gpu_lib.ce_fwd_bwd_f32(z, t, 1.0, ws=ws) for _ in range(3)]
    for loss, dz in a[1:]:
        assert torch.equal(loss, a[0][0]) and torch.equal(dz, a[0][1])
    # the forward-only call gives the same loss bits
    assert torch.equal(gpu_lib.ce_fwd_f32(z, t, ws=ws), a[0][0]) or \
        float(gpu_lib.ce_fwd_f32(z, t, ws=ws).item()) == pytest.approx(float(a[0][0].item()), rel=1e-6)


@pytest.mark.parametrize("V", [4096, 131072])
def test_flat_full_size_sampled_rows(gpu_lib, V):
    """fp32 [16384, V] ~ N(0,1): loss against the kernel's own rows, gradient
    rows sampled and compared with the oracle on rows regenerated on the host."""
    T = 16384
    z = gen.normal_f32(0, gen.STREAM_LOGITS, (T, V))
    t = gen.targets(0, gen.STREAM_TARGET, (T,), V)
    m, rows, dz = run_flat(gpu_lib, z, t, 1.0)
    idx = sample_rows(T, 16)
    _, rows_ref = oracle.ce_f32(z[idx], t[idx])
    np.testing.assert_allclose(rows[idx], rows_ref, rtol=1e-5, atol=1e-6)
    got = dz[torch.from_numpy(idx).cuda()].cpu().numpy()
    ref = oracle.ce_grad_f64(z[idx].astype(np.float64), t[idx], None, 1.0 / T)
    np.testing.assert_allclose(got, ref, rtol=2e-5, atol=1e-7 / T)


SBV = [(1, 1, 1), (3, 2, 5), (16, 4, 8193), (2, 4, 32768), (3, 1, 131072), (700, 4, 2048)]


@pytest.mark.parametrize("with_dloss", [False, True])
@pytest.mark.parametrize("S,B,V", SBV)
def test_sbv_fwd_bwd_matches_oracle(gpu_lib, S, B, V, with_dloss):
    zb = gen.normal_bf16_bits(34, 0, (S, B, V), sigma=2.0)
    t = gen.targets(34, 1, (S, B), V)
    dl = gen.normal_f32(34, 5, (S, B)) if with_dloss else None
    loss, dz = gpu_lib.ce_fwd_bwd_sbv_bf16(to_dev_bf16(zb), to_dev(t), None if dl is None else to_dev(dl), 0.5)
    torch.cuda.synchronize()
    np.testing.assert_allclose(loss.cpu().numpy(), oracle.ce_sbv_bf16(zb, t), rtol=0, atol=2e-3)
    ref = oracle.ce_grad_sbv_bf16(zb, t, None if dl is None else dl.astype(np.float64), 0.5)
    gmax = 0.5 * (1.0 if dl is None else float(np.abs(dl).max()))
    np.testing.assert_allclose(bf16_to_f64(dz), ref, rtol=4.5e-3, atol=1e-7 * gmax)


def test_sbv_full_size_sampled(gpu_lib):
    S, B, V = 2048, 4, 32768
    zb = gen.normal_bf16_bits(0, gen.STREAM_LOGITS, (S, B, V), sigma=2.0)
    t = gen.targets(0, gen.STREAM_TARGET, (S, B), V)
    loss, dz = gpu_lib.ce_fwd_bwd_sbv_bf16(to_dev_bf16(zb), to_dev(t))
    idx = sample_rows(S * B, 12)
    got = bf16_to_f64(dz.view(S * B, V)[torch.from_numpy(idx).cuda()])
    zr = zb.reshape(S * B, 1, V)[idx]
    ref = oracle.ce_grad_sbv_bf16(zr, t.reshape(-1, 1)[idx]).reshape(len(idx), V)
    np.testing.assert_allclose(got, ref, rtol=4.5e-3, atol=1e-7)
    np.testing.assert_allclose(loss.cpu().numpy().reshape(-1)[idx],
                               oracle.ce_sbv_bf16(zr, t.reshape(-1, 1)[idx]).reshape(-1), rtol=0, atol=2e-3)


def test_fwd_bwd_argument_errors(gpu_lib):
    z = torch.zeros((4, 8), device="cuda")
    t = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(gpu_lib.LmhoError) as e:
        gpu_lib.ce_fwd_bwd_f32(z, t, dlogits=z)          # gradient over the logits
    assert e.value.status == gpu_lib.LMHO_ERR_ALIAS
    with pytest.raises(gpu_lib.LmhoError) as e:
        gpu_lib.ce_fwd_bwd_f32(z, t, grad_scale=float("inf"))
    assert e.value.status == gpu_lib.LMHO_ERR_INVALID_ARG


@pytest.mark.parametrize("T,V", [(301, 2048), (5, 512), (7, 4096), (3, 2052)])
def test_flat_warp_rows_bad_targets_and_odd_rows(gpu_lib, T, V):
    # aligned rows of at most 16 KB take the warp-per-row kernel (two warps per
    # row above 8 KB): an odd row count leaves one warp of the last block idle
    # (one warp per row); targets out of range on
    # either side make their rows (loss and gradient) NaN and the mean NaN
    z = gen.normal_f32(35, 0, (T, V))
    t = gen.targets(35, 1, (T,), V)
    t[0], t[T - 1] = -1, V
    m, rows, dz = run_flat(gpu_lib, z, t, 0.75)
    d = dz.cpu().numpy().astype(np.float64)
    assert math.isnan(m) and np.isnan(rows[0]) and np.isnan(rows[T - 1])
    assert np.all(np.isnan(d[0])) and np.all(np.isnan(d[T - 1]))
    keep = np.arange(1, T - 1)
    rows_ref = oracle.ce_f32(z[keep], t[keep])[1]
    np.testing.assert_allclose(rows[keep], rows_ref, rtol=1e-5, atol=1e-6)
    ref = oracle.ce_grad_f32(z[keep], t[keep], 0.75) * (len(keep) / T)
    np.testing.assert_allclose(d[keep], ref, rtol=2e-5, atol=1e-7 * 0.75 / T)


@pytest.mark.parametrize("S,B,V", [(3, 3, 4096), (5, 1, 8), (3, 3, 8192), (1, 3, 4104)])
def test_sbv_warp_rows_bad_targets_and_odd_rows(gpu_lib, S, B, V):
    zb = gen.normal_bf16_bits(36, 0, (S, B, V), sigma=2.0)
    t = gen.targets(36, 1, (S, B), V)
    dl = gen.normal_f32(36, 5, (S, B))
    t[0, 0], t[S - 1, B - 1] = -7, V + 3
    loss, dz = gpu_lib.ce_fwd_bwd_sbv_bf16(to_dev_bf16(zb), to_dev(t), to_dev(dl), 0.5)
    torch.cuda.synchronize()
    lo = loss.cpu().numpy().reshape(-1)
    d = bf16_to_f64(dz).reshape(S * B, V)
    assert np.isnan(lo[0]) and np.isnan(lo[-1]) and np.all(np.isnan(d[0])) and np.all(np.isnan(d[-1]))
    keep = np.arange(1, S * B - 1)
    zr = zb.reshape(S * B, 1, V)[keep]
    tr = t.reshape(-1, 1)[keep]
    np.testing.assert_allclose(lo[keep], oracle.ce_sbv_bf16(zr, tr).reshape(-1), rtol=0, atol=2e-3)
    ref = oracle.ce_grad_sbv_bf16(zr, tr, dl.reshape(-1, 1)[keep].astype(np.float64), 0.5).reshape(len(keep), V)
    gmax = 0.5 * float(np.abs(dl).max())
    np.testing.assert_allclose(d[keep], ref, rtol=4.5e-3, atol=1e-7 * gmax)
