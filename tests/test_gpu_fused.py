"""GPU parity of the tensor-core fused-linear kernels against the fp64 oracle.

Pages "Fused linear + CPO loss" (its cross-entropy core: x [batch*seq,
hidden] through a vocab x hidden head, integer targets, mean loss[1], logits
never materialised) and "Fused linear + JSD" (student/teacher heads,
generalized JSD, batchmean).  Bar: relative error <= 2e-3 on the scalars.
Per-token values are held tighter (1e-4 relative on CE losses; 1e-3
relative + 1e-5 absolute on per-token JSD), which the fp32 tensor-core
accumulation of exact bf16 products comfortably meets.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.helpers import tile_samples, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

RTOL_SCALAR = 2e-3
RTOL_CE_TOKEN = 1e-4
RTOL_JSD_TOKEN, ATOL_JSD_TOKEN = 1e-3, 1e-5


def flce_inputs(seed, T, H, V, sw=0.02):
    x = gen.normal_bf16_bits(seed, gen.STREAM_X, (T, H))
    W = gen.normal_bf16_bits(seed, gen.STREAM_W, (V, H), sigma=sw)
    t = gen.targets(seed, gen.STREAM_TARGET, (T,), V)
    return x, W, t


def run_flce(lmho, x, W, t):
    T, H = x.shape
    V = W.shape[0]
    ws = lmho.workspace(lmho.flce_workspace_bytes(T, H, V))
    loss = lmho.flce_fwd_bf16(to_dev_bf16(x), to_dev_bf16(W), to_dev(t), ws=ws)
    assert lmho.ws_status(ws) == 0
    return float(loss.item()), lmho.row_losses(ws, T).cpu().numpy().astype(np.float64)


FLCE_SHAPES = [(1, 64, 1), (5, 64, 37), (128, 64, 256), (130, 128, 1000), (257, 200, 4097), (64, 1024, 513),
               (300, 4096, 777), (1, 4096, 128256)]


@pytest.mark.parametrize("T,H,V", FLCE_SHAPES)
def test_flce_matches_oracle(gpu_lib, T, H, V):
    # sigma_w = 2/sqrt(H) keeps logits O(1) at every H
    x, W, t = flce_inputs(7, T, H, V, sw=2.0 / math.sqrt(H))
    m, rows = run_flce(gpu_lib, x, W, t)
    m_ref, rows_ref = oracle.flce_bf16(x, W, t)
    np.testing.assert_allclose(rows, rows_ref, rtol=RTOL_CE_TOKEN, atol=1e-5)
    assert m == pytest.approx(m_ref, rel=RTOL_SCALAR)


def test_flce_zero_input_is_ln_V_and_deterministic(gpu_lib):
    T, H, V = 200, 128, 3000
    x = np.zeros((T, H), np.uint16)
    _, W, t = flce_inputs(8, T, H, V)
    m, rows = run_flce(gpu_lib, x, W, t)
    np.testing.assert_allclose(rows, math.log(V), rtol=1e-6)
    x, W, t = flce_inputs(8, T, H, V, sw=0.1)
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    ws = gpu_lib.workspace(gpu_lib.flce_workspace_bytes(T, H, V))
    first = gpu_lib.flce_fwd_bf16(xd, Wd, td, ws=ws).clone()
    for _ in range(4):
        assert torch.equal(gpu_lib.flce_fwd_bf16(xd, Wd, td, ws=ws), first)


def test_raster_group_changes_order_not_results(gpu_lib):
    """The unit order (raster group) must not change a single bit: each
    (token tile, vocab tile) partial is computed the same way in any order."""
    T, H, V = 1100, 256, 5000
    x, W, t = flce_inputs(14, T, H, V, sw=0.1)
    xs, Ws, xt, Wt = jsd_inputs(14, T, H, V, sw=0.1)
    outs = []
    try:
        for g in (1, 3, 16, 64):
            gpu_lib.set_raster_group(g)
            outs.append((run_flce(gpu_lib, x, W, t), run_fljsd(gpu_lib, xs, Ws, xt, Wt)))
    finally:
        gpu_lib.set_raster_group(0)
    for (fl, js) in outs[1:]:
        assert fl[0] == outs[0][0][0] and np.array_equal(fl[1], outs[0][0][1])
        assert js[0] == outs[0][1][0] and np.array_equal(js[1], outs[0][1][1])


def test_flce_bad_target_gives_nan(gpu_lib):
    T, H, V = 10, 64, 300
    x, W, t = flce_inputs(9, T, H, V)
    t[3] = V
    t[4] = -5
    m, rows = run_flce(gpu_lib, x, W, t)
    assert np.isnan(rows[3]) and np.isnan(rows[4]) and math.isnan(m)
    assert np.all(np.isfinite(np.delete(rows, [3, 4])))


@pytest.mark.parametrize("batch", [2, 16])
def test_flce_full_size_sampled(gpu_lib, batch):
    """x bf16 [batch*1024, 4096] ~ N(0,1), W bf16 [128256, 4096] ~ N(0, 0.02^2):
    one token of every 128-token tile, the last token and both sides of every
    raster-group boundary (groups of 32 tiles) against the oracle; mean
    against the kernel's own per-token losses and the closed-form expectation
    ln V + H sigma_w^2 / 2."""
    T, H, V = batch * 1024, 4096, 128256
    x, W, t = flce_inputs(0, T, H, V)
    m, rows = run_flce(gpu_lib, x, W, t)
    idx = tile_samples(T, groups=(32,), seed=batch)
    _, ref = oracle.flce_bf16(x[idx], W, t[idx])
    np.testing.assert_allclose(rows[idx], ref, rtol=RTOL_CE_TOKEN, atol=1e-5)
    assert m == pytest.approx(rows.mean(), rel=1e-6)
    assert abs(m - (math.log(V) + H * 0.02 ** 2 / 2)) < 0.05


# ---------------------------------------------------------------- JSD
def jsd_inputs(seed, T, H, V, sw=0.02):
    xs = gen.normal_bf16_bits(seed, gen.STREAM_X, (T, H))
    Ws = gen.normal_bf16_bits(seed, gen.STREAM_W, (V, H), sigma=sw)
    xt = gen.normal_bf16_bits(seed, gen.STREAM_XT, (T, H))
    Wt = gen.normal_bf16_bits(seed, gen.STREAM_WT, (V, H), sigma=sw)
    return xs, Ws, xt, Wt


def run_fljsd(lmho, xs, Ws, xt, Wt, beta=0.5):
    T, H = xs.shape
    V = Ws.shape[0]
    ws = lmho.workspace(lmho.fljsd_workspace_bytes(T, H, V))
    loss = lmho.fljsd_fwd_bf16(to_dev_bf16(xs), to_dev_bf16(Ws), to_dev_bf16(xt), to_dev_bf16(Wt), beta, ws=ws)
    assert lmho.ws_status(ws) == 0
    return float(loss.item()), lmho.row_losses(ws, T).cpu().numpy().astype(np.float64)


JSD_SHAPES = [(1, 64, 2), (5, 64, 37), (130, 128, 1000), (64, 256, 4097), (129, 4096, 300)]


@pytest.mark.parametrize("beta", [0.5, 0.3])
@pytest.mark.parametrize("T,H,V", JSD_SHAPES)
def test_fljsd_matches_oracle(gpu_lib, T, H, V, beta):
    xs, Ws, xt, Wt = jsd_inputs(10, T, H, V, sw=2.0 / math.sqrt(H))
    m, rows = run_fljsd(gpu_lib, xs, Ws, xt, Wt, beta)
    m_ref, rows_ref = oracle.fljsd_bf16(xs, Ws, xt, Wt, beta)
    np.testing.assert_allclose(rows, rows_ref, rtol=RTOL_JSD_TOKEN, atol=ATOL_JSD_TOKEN)
    assert m == pytest.approx(m_ref, rel=RTOL_SCALAR)


def test_fljsd_identical_heads_is_zero(gpu_lib):
    T, H, V = 70, 128, 2000
    xs, Ws, _, _ = jsd_inputs(11, T, H, V, sw=0.2)
    m, rows = run_fljsd(gpu_lib, xs, Ws, xs, Ws)
    assert abs(m) <= 1e-6 and np.all(np.abs(rows) <= 1e-6)


def test_fljsd_bounds_and_symmetry(gpu_lib):
    T, H, V = 64, 128, 1500
    xs, Ws, xt, Wt = jsd_inputs(12, T, H, V, sw=0.3)
    m1, r1 = run_fljsd(gpu_lib, xs, Ws, xt, Wt)
    m2, r2 = run_fljsd(gpu_lib, xt, Wt, xs, Ws)
    assert np.all(r1 >= -1e-6) and np.all(r1 <= math.log(2) + 1e-6)
    np.testing.assert_allclose(r1, r2, rtol=1e-4, atol=1e-6)
    # beta <-> 1 - beta with the heads swapped is the same divergence
    m3, _ = run_fljsd(gpu_lib, xs, Ws, xt, Wt, 0.2)
    m4, _ = run_fljsd(gpu_lib, xt, Wt, xs, Ws, 0.8)
    assert m3 == pytest.approx(m4, rel=1e-4)


@pytest.mark.parametrize("T", [1024, 8192])
def test_fljsd_full_size_sampled(gpu_lib, T):
    """Student/teacher bf16 [T, 4096] ~ N(0,1), heads [128256, 4096] ~ N(0, 0.02^2),
    beta 0.5: one token of every 128-token tile, the last token and both sides
    of every raster-group boundary of both passes (16 and 32 tiles) against
    the oracle."""
    H, V = 4096, 128256
    xs, Ws, xt, Wt = jsd_inputs(0, T, H, V)
    m, rows = run_fljsd(gpu_lib, xs, Ws, xt, Wt)
    idx = tile_samples(T, groups=(16, 32), seed=T)
    _, ref = oracle.fljsd_bf16(xs[idx], Ws, xt[idx], Wt, 0.5)
    np.testing.assert_allclose(rows[idx], ref, rtol=RTOL_JSD_TOKEN, atol=ATOL_JSD_TOKEN)
    assert m == pytest.approx(rows.mean(), rel=1e-6)
    assert 0.0 < m < math.log(2)


def test_wait_timeout_reports_status(gpu_lib):
    """A bounded in-kernel wait on a barrier nothing completes gives up and
    reports LMHO_ERR_TIMEOUT through the workspace status word; the context
    stays usable."""
    ws = gpu_lib.workspace(256)
    gpu_lib.selftest_wait_timeout(ws, 2_000_000)   # 2 ms
    assert gpu_lib.ws_status(ws) == gpu_lib.LMHO_ERR_TIMEOUT
    assert gpu_lib.ws_status(ws) == 0               # cleared by the read
    x, W, t = flce_inputs(13, 8, 64, 100)
    m, rows = run_flce(gpu_lib, x, W, t)
    assert np.all(np.isfinite(rows))


# ---------------------------------------------------------------- JSD variant: temperature, token mask
def run_fljsd_ex(lmho, xs, Ws, xt, Wt, beta, tau, keep):
    T, H = xs.shape
    V = Ws.shape[0]
    ws = lmho.workspace(lmho.fljsd_workspace_bytes(T, H, V))
    kd = None if keep is None else to_dev(keep)
    loss = lmho.fljsd_fwd_bf16_ex(to_dev_bf16(xs), to_dev_bf16(Ws), to_dev_bf16(xt), to_dev_bf16(Wt), beta, tau, kd,
                                  ws=ws)
    assert lmho.ws_status(ws) == 0
    return float(loss.item()), lmho.row_losses(ws, T).cpu().numpy().astype(np.float64)


def test_fljsd_ex_defaults_are_bitwise_base(gpu_lib):
    xs, Ws, xt, Wt = jsd_inputs(16, 300, 128, 3000, sw=0.2)
    a = run_fljsd(gpu_lib, xs, Ws, xt, Wt, 0.4)
    b = run_fljsd_ex(gpu_lib, xs, Ws, xt, Wt, 0.4, 1.0, None)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("tau,beta", [(2.0, 0.5), (0.7, 0.3), (4.0, 0.5)])
@pytest.mark.parametrize("T,H,V", [(130, 128, 1000), (7, 4096, 2049)])
def test_fljsd_ex_temperature_and_mask_match_oracle(gpu_lib, tau, beta, T, H, V):
    xs, Ws, xt, Wt = jsd_inputs(17, T, H, V, sw=2.0 / math.sqrt(H))
    keep = (gen.targets(17, 1, (T,), 3) != 0).astype(np.uint8)   # about two thirds kept
    for k in (None, keep):
        m, rows = run_fljsd_ex(gpu_lib, xs, Ws, xt, Wt, beta, tau, k)
        m_ref, rows_ref = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, beta, tau, k)
        np.testing.assert_allclose(rows, rows_ref, rtol=RTOL_JSD_TOKEN, atol=ATOL_JSD_TOKEN)
        assert m == pytest.approx(m_ref, rel=RTOL_SCALAR)


def test_fljsd_ex_nothing_kept_is_zero(gpu_lib):
    xs, Ws, xt, Wt = jsd_inputs(18, 40, 64, 500, sw=0.3)
    m, rows = run_fljsd_ex(gpu_lib, xs, Ws, xt, Wt, 0.5, 1.0, np.zeros(40, np.uint8))
    assert m == 0.0 and np.all(rows == 0.0)
