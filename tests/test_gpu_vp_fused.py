"""GPU parity of the vocab-parallel fused losses against the fp64 oracle.

The vocabulary split of the page "Vocab-parallel cross-entropy, Megatron
layout" (summary: each tensor-parallel rank holds its own vocab range) applied
to the output layer of the fused losses (pages "Fused linear + CPO loss", its
cross-entropy core, and "Fused linear + JSD"): a rank holds the rows
[v0, v0 + V_local) of W.  The ranks are emulated on one GPU: W is cut into k
uneven row blocks, each copied to its own buffer (a rank's local head); the
per-shard results are stacked as an all-gather in rank order leaves them and
merged by the library's merge calls.

Bars: as the unsharded fused tests (per-token CE losses 1e-4 relative;
per-token JSD 1e-3 relative + 1e-5 absolute; scalars 2e-3 relative).  Shard
log-sum-exps 1e-5 relative.  With one shard (the whole W) every result must
equal the unsharded call's bit for bit: the merges of a single block are
exact and every other step is the same kernel.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.helpers import assert_within_bounds, ce_error_scale, grad_bounds, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

RTOL_SCALAR = 2e-3
RTOL_CE_TOKEN = 1e-4
RTOL_JSD_TOKEN, ATOL_JSD_TOKEN = 1e-3, 1e-5
RTOL_LSE = 1e-5


def uneven_shards(V, k, seed):
    if k == 1:
        return [(0, V)]
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, V), size=k - 1, replace=False))
    edges = np.concatenate([[0], cuts, [V]])
    return [(int(a), int(b - a)) for a, b in zip(edges[:-1], edges[1:])]


def flce_inputs(seed, T, H, V):
    x = gen.normal_bf16_bits(seed, gen.STREAM_X, (T, H))
    W = gen.normal_bf16_bits(seed, gen.STREAM_W, (V, H), sigma=2.0 / math.sqrt(H))
    t = gen.targets(seed, gen.STREAM_TARGET, (T,), V)
    return x, W, t


def jsd_inputs(seed, T, H, V, sw):
    xs = gen.normal_bf16_bits(seed, gen.STREAM_X, (T, H))
    Ws = gen.normal_bf16_bits(seed, gen.STREAM_W, (V, H), sigma=sw)
    xt = gen.normal_bf16_bits(seed, gen.STREAM_XT, (T, H))
    Wt = gen.normal_bf16_bits(seed, gen.STREAM_WT, (V, H), sigma=sw)
    return xs, Ws, xt, Wt


def run_flce_vp(lmho, xd, Wd, td, shards, V):
    """Returns (partials [k, 3, T], per-token losses [T], mean [1])."""
    T = xd.shape[0]
    parts = torch.full((len(shards), 3, T), float("nan"), device="cuda")
    for j, (v0, w) in enumerate(shards):
        lmho.flce_partials_bf16(xd, Wd[v0:v0 + w].clone(), td, v0, partials=parts[j])
    rows = lmho.ce_merge_partials(parts.view(len(shards), 3, T, 1), td.view(T, 1), V).view(T)
    mean = lmho.rows_mean(rows)
    torch.cuda.synchronize()
    return parts, rows, mean


def run_fljsd_vp(lmho, xsd, Wsd, xtd, Wtd, shards, beta, tau, keep=None):
    """Returns (lse parts [k, 2, T], lse [2, T], terms [k, T], rows [T], loss [1])."""
    T = xsd.shape[0]
    k = len(shards)
    local = [(Wsd[v0:v0 + w].clone(), Wtd[v0:v0 + w].clone()) for v0, w in shards]
    lparts = torch.full((k, 2, T), float("nan"), device="cuda")
    for j, (a, b) in enumerate(local):
        lmho.fljsd_lse_partials_bf16(xsd, a, xtd, b, tau, out=lparts[j])
    lse = lmho.lse_merge_partials(lparts)
    terms = torch.full((k, T), float("nan"), device="cuda")
    for j, (a, b) in enumerate(local):
        lmho.fljsd_terms_bf16(xsd, a, xtd, b, lse, beta, tau, out=terms[j])
    loss, rows = lmho.jsd_merge_terms(terms, keep)
    torch.cuda.synchronize()
    return lparts, lse, terms, rows, loss


def np64(t):
    return t.cpu().numpy().astype(np.float64)


# ---------------------------------------------------------------- fused linear + CE
FLCE_VP_CASES = [(64, 64, 300, 2), (200, 128, 1500, 3), (129, 256, 777, 4), (5, 64, 37, 5), (96, 4096, 2000, 3)]


@pytest.mark.parametrize("T,H,V,k", FLCE_VP_CASES)
def test_flce_vp_matches_oracle(gpu_lib, T, H, V, k):
    x, W, t = flce_inputs(20 + k, T, H, V)
    shards = uneven_shards(V, k, 3 + k)
    # targets on every shard's first and last column, then one out of range each way
    edge = [c for v0, w in shards for c in (v0, v0 + w - 1)]
    n = min(len(edge), T - 2) if T > 2 else 0
    t[:n] = edge[:n]
    if T > 2:
        t[-2], t[-1] = -1, V
    parts, rows, mean = run_flce_vp(gpu_lib, to_dev_bf16(x), to_dev_bf16(W), to_dev(t), shards, V)
    # per shard: the shard log-sum-exp m + ln s, and the target logit or -inf
    for j, (v0, w) in enumerate(shards):
        m, s, zt = oracle.flce_partials_bf16(x, np.ascontiguousarray(W[v0:v0 + w]), t, v0)
        p = np64(parts[j])
        np.testing.assert_allclose(p[0] + np.log(p[1]), m + np.log(s), rtol=RTOL_LSE, atol=1e-5)
        own = (t >= v0) & (t < v0 + w)
        assert np.all(p[2][~own] == -np.inf)
        np.testing.assert_allclose(p[2][own], zt[own], rtol=1e-5, atol=1e-5)
    _, want = oracle.flce_bf16(x, W, t)
    got = np64(rows)
    bad = (t < 0) | (t >= V)
    assert np.all(np.isnan(got[bad])) and np.all(np.isnan(want[bad]))
    np.testing.assert_allclose(got[~bad], want[~bad], rtol=RTOL_CE_TOKEN, atol=1e-5)
    if not bad.any():
        assert float(mean.item()) == pytest.approx(want.mean(), rel=RTOL_SCALAR)


def test_flce_vp_mean_and_single_shard_bitwise(gpu_lib):
    """One shard holding all of W gives flce_fwd_bf16's per-token losses and
    mean bit for bit; three shards give the same within rounding."""
    T, H, V = 300, 256, 3000
    x, W, t = flce_inputs(31, T, H, V)
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    ws = gpu_lib.workspace(gpu_lib.flce_workspace_bytes(T, H, V))
    ref = gpu_lib.flce_fwd_bf16(xd, Wd, td, ws=ws)
    ref_rows = gpu_lib.row_losses(ws, T).clone()
    _, rows1, mean1 = run_flce_vp(gpu_lib, xd, Wd, td, [(0, V)], V)
    assert torch.equal(rows1, ref_rows) and torch.equal(mean1, ref)
    _, rows3, mean3 = run_flce_vp(gpu_lib, xd, Wd, td, uneven_shards(V, 3, 1), V)
    torch.testing.assert_close(rows3, ref_rows, rtol=1e-5, atol=1e-5)
    assert float(mean3.item()) == pytest.approx(float(ref.item()), rel=1e-5)


def test_flce_vp_deterministic(gpu_lib):
    T, H, V = 257, 128, 1000
    x, W, t = flce_inputs(33, T, H, V)
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    shards = uneven_shards(V, 3, 7)
    a = run_flce_vp(gpu_lib, xd, Wd, td, shards, V)
    b = run_flce_vp(gpu_lib, xd, Wd, td, shards, V)
    assert all(torch.equal(p, q) for p, q in zip(a, b))


def test_flce_vp_full_size_sampled(gpu_lib):
    """x [2048, 4096], W [128256, 4096] ~ N(0, 0.02^2) split over 8 ranks
    (16032 rows each, as tensor parallelism 8 would): the merged losses within
    1e-5 of the unsharded call and sampled tokens against the oracle."""
    T, H, V, k = 2048, 4096, 128256, 8
    x = gen.normal_bf16_bits(0, gen.STREAM_X, (T, H))
    W = gen.normal_bf16_bits(0, gen.STREAM_W, (V, H), sigma=0.02)
    t = gen.targets(0, gen.STREAM_TARGET, (T,), V)
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    shards = [(j * V // k, (j + 1) * V // k - j * V // k) for j in range(k)]
    _, rows, mean = run_flce_vp(gpu_lib, xd, Wd, td, shards, V)
    ws = gpu_lib.workspace(gpu_lib.flce_workspace_bytes(T, H, V))
    ref = gpu_lib.flce_fwd_bf16(xd, Wd, td, ws=ws)
    torch.testing.assert_close(rows, gpu_lib.row_losses(ws, T), rtol=1e-5, atol=1e-5)
    assert float(mean.item()) == pytest.approx(float(ref.item()), rel=1e-5)
    idx = np.array([0, 1, 127, 128, 1023, 1024, 2046, 2047])
    _, want = oracle.flce_bf16(x[idx], W, t[idx])
    np.testing.assert_allclose(np64(rows)[idx], want, rtol=RTOL_CE_TOKEN, atol=1e-5)


# ---------------------------------------------------------------- fused linear + CE backward of a shard
def run_flce_vp_bwd(lmho, xd, Wd, td, shards, V, scale):
    """Forward partials of every shard, then each shard's backward with the
    gathered partials: returns (partials [k, 3, T], [(dx share, dW rows)])."""
    parts, _, _ = run_flce_vp(lmho, xd, Wd, td, shards, V)
    outs = [lmho.flce_shard_bwd_bf16(xd, Wd[v0:v0 + w].clone(), td, parts, v0, V, scale) for v0, w in shards]
    torch.cuda.synchronize()
    return parts, outs


@pytest.mark.parametrize("T,H,V,k", [(130, 128, 1000, 3), (257, 200, 4097, 2), (64, 256, 513, 4),
                                     (96, 1024, 2000, 3)])
def test_flce_vp_backward_matches_oracle(gpu_lib, T, H, V, k):
    """Each shard's dx share and dW rows against the oracle's shard gradient,
    every element within its own bound (bf16 dZ, fp32 accumulation over the
    shard's K); the shares' sum against the unsharded oracle dx within the
    sum of the shares' bounds."""
    x, W, t = flce_inputs(70 + k, T, H, V)
    shards = uneven_shards(V, k, 12 + k)
    edge = [c for v0, w in shards for c in (v0, v0 + w - 1)]
    t[:min(T, len(edge))] = edge[:T]
    scale = 1.3
    _, outs = run_flce_vp_bwd(gpu_lib, to_dev_bf16(x), to_dev_bf16(W), to_dev(t), shards, V, scale)
    dz = oracle.ce_grad_f64(oracle.logits_bf16(x, W), t, None, scale / T)
    S = ce_error_scale(dz, t, scale / T)
    xd = gen.bf16_bits_to_f32(x).astype(np.float64)
    Wd = gen.bf16_bits_to_f32(W).astype(np.float64)
    om = [oracle.flce_partials_bf16(x, np.ascontiguousarray(W[v0:v0 + w]), t, v0) for v0, w in shards]
    lse = oracle.ce_partials_lse(np.stack([p[0] for p in om]), np.stack([p[1] for p in om]))
    dx_sum, b_sum = np.zeros((T, H)), np.zeros((T, H))
    for j, (v0, w) in enumerate(shards):
        bdx, bdW = grad_bounds(dz[:, v0:v0 + w], S[:, v0:v0 + w], xd, Wd[v0:v0 + w])
        dx_ref, dW_ref = oracle.flce_grad_shard_bf16(x, np.ascontiguousarray(W[v0:v0 + w]), t, v0, V, lse, scale)
        got_dx, got_dW = np64(outs[j][0]), np64(outs[j][1])
        assert_within_bounds(got_dx, dx_ref, bdx, f"dx share of shard {j}")
        assert_within_bounds(got_dW, dW_ref, bdW, f"dW rows of shard {j}")
        dx_sum += got_dx
        b_sum += bdx
    dx_full, _ = oracle.flce_grad_bf16(x, W, t, scale)
    assert_within_bounds(dx_sum, dx_full, b_sum, "sum of the dx shares")


def test_flce_vp_backward_single_shard_bitwise_and_bad_target(gpu_lib):
    """One shard holding all of W gives flce_fwd_bwd_bf16's dx and dW bit for
    bit; a target outside [0, V) gives a NaN dx row and NaN dW, as unsharded."""
    T, H, V = 200, 256, 3000
    x, W, t = flce_inputs(75, T, H, V)
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    ws = gpu_lib.workspace(gpu_lib.flce_bwd_workspace_bytes(T, H, V))
    _, dx_ref, dW_ref = gpu_lib.flce_fwd_bwd_bf16(xd, Wd, td, 0.7, ws=ws)
    _, outs = run_flce_vp_bwd(gpu_lib, xd, Wd, td, [(0, V)], V, 0.7)
    assert torch.equal(outs[0][0], dx_ref) and torch.equal(outs[0][1], dW_ref)
    t[5] = V
    _, outs = run_flce_vp_bwd(gpu_lib, xd, Wd, to_dev(t), uneven_shards(V, 2, 3), V, 0.7)
    for dx, dW in outs:
        assert bool(torch.isnan(dx[5]).all()) and bool(torch.isfinite(torch.cat([dx[:5], dx[6:]])).all())
        assert bool(torch.isnan(dW).all())


def test_flce_vp_backward_full_size(gpu_lib):
    """x [2048, 4096], W [128256, 4096] ~ N(0, 0.02^2) over 8 shards: the dx
    shares' sum and the stacked dW rows against the unsharded backward
    (normwise 1e-3: both round dZ to bf16 from normalisers merged in different
    orders), and sampled dx rows against the oracle within their bounds."""
    T, H, V, k = 2048, 4096, 128256, 8
    x = gen.normal_bf16_bits(0, gen.STREAM_X, (T, H))
    W = gen.normal_bf16_bits(0, gen.STREAM_W, (V, H), sigma=0.02)
    t = gen.targets(0, gen.STREAM_TARGET, (T,), V)
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    shards = [(j * V // k, (j + 1) * V // k - j * V // k) for j in range(k)]
    _, outs = run_flce_vp_bwd(gpu_lib, xd, Wd, td, shards, V, 1.0)
    dx = outs[0][0].clone()
    for j in range(1, k):
        dx += outs[j][0]
    dW = torch.cat([o[1] for o in outs])
    del outs
    ws = gpu_lib.workspace(gpu_lib.flce_bwd_workspace_bytes(T, H, V))
    _, dx_ref, dW_ref = gpu_lib.flce_fwd_bwd_bf16(xd, Wd, td, 1.0, ws=ws)
    assert float(torch.linalg.norm(dx - dx_ref)) <= 1e-3 * float(torch.linalg.norm(dx_ref))
    assert float(torch.linalg.norm(dW - dW_ref)) <= 1e-3 * float(torch.linalg.norm(dW_ref))
    del dW, dW_ref, ws
    idx = np.array([0, 777, 2047])
    dz = oracle.ce_grad_f64(oracle.logits_bf16(x[idx], W), t[idx], None, 1.0 / T)
    S = ce_error_scale(dz, t[idx], 1.0 / T)
    Wd64 = gen.bf16_bits_to_f32(W).astype(np.float64)
    bdx, _ = grad_bounds(dz, S, gen.bf16_bits_to_f32(x[idx]).astype(np.float64), Wd64)
    assert_within_bounds(np64(dx)[idx], dz @ Wd64, bdx, "dx rows (sum of 8 shares)")


# ---------------------------------------------------------------- fused linear + JSD
FLJSD_VP_CASES = [(64, 64, 300, 2, 0.5, 1.0, False), (200, 128, 1500, 3, 0.3, 2.0, True),
                  (129, 256, 777, 4, 0.5, 0.7, False), (5, 64, 37, 5, 0.8, 1.0, True),
                  (64, 4096, 2000, 3, 0.5, 1.0, False)]


@pytest.mark.parametrize("T,H,V,k,beta,tau,masked", FLJSD_VP_CASES)
def test_fljsd_vp_matches_oracle(gpu_lib, T, H, V, k, beta, tau, masked):
    xs, Ws, xt, Wt = jsd_inputs(40 + k, T, H, V, sw=2.0 / math.sqrt(H))
    keep = (np.arange(T) % 4 != 2).astype(np.uint8) if masked else None
    shards = uneven_shards(V, k, 9 + k)
    lparts, lse, terms, rows, loss = run_fljsd_vp(gpu_lib, to_dev_bf16(xs), to_dev_bf16(Ws), to_dev_bf16(xt),
                                                  to_dev_bf16(Wt), shards, beta, tau,
                                                  None if keep is None else to_dev(keep))
    sl = [(np.ascontiguousarray(Ws[v0:v0 + w]), np.ascontiguousarray(Wt[v0:v0 + w])) for v0, w in shards]
    want_parts = np.stack([oracle.fljsd_lse_shard_bf16(xs, a, xt, b, tau) for a, b in sl])
    np.testing.assert_allclose(np64(lparts), want_parts, rtol=RTOL_LSE, atol=1e-5)
    want_lse = oracle.lse_merge(want_parts)
    np.testing.assert_allclose(np64(lse), want_lse, rtol=RTOL_LSE, atol=1e-5)
    want_terms = np.stack([oracle.fljsd_terms_shard_bf16(xs, a, xt, b, want_lse, beta, tau) for a, b in sl])
    np.testing.assert_allclose(np64(terms), want_terms, rtol=RTOL_JSD_TOKEN, atol=ATOL_JSD_TOKEN)
    want_mean, want_rows = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, beta, tau, keep)
    np.testing.assert_allclose(np64(rows), want_rows, rtol=RTOL_JSD_TOKEN, atol=ATOL_JSD_TOKEN)
    if keep is not None:
        assert np.all(np64(rows)[keep == 0] == 0.0)
    assert float(loss.item()) == pytest.approx(want_mean, rel=RTOL_SCALAR)


@pytest.mark.parametrize("beta,tau,masked", [(0.5, 1.0, False), (0.3, 2.0, True)])
def test_fljsd_vp_single_shard_is_bitwise_unsharded(gpu_lib, beta, tau, masked):
    T, H, V = 300, 128, 3000
    xs, Ws, xt, Wt = jsd_inputs(51, T, H, V, sw=0.2)
    d = [to_dev_bf16(a) for a in (xs, Ws, xt, Wt)]
    keep = to_dev((np.arange(T) % 3 != 0).astype(np.uint8)) if masked else None
    ws = gpu_lib.workspace(gpu_lib.fljsd_workspace_bytes(T, H, V))
    ref = gpu_lib.fljsd_fwd_bf16_ex(*d, beta, tau, keep, ws=ws)
    ref_rows = gpu_lib.row_losses(ws, T).clone()
    _, _, _, rows, loss = run_fljsd_vp(gpu_lib, *d, [(0, V)], beta, tau, keep)
    assert torch.equal(rows, ref_rows) and torch.equal(loss, ref)
    _, _, _, rows3, loss3 = run_fljsd_vp(gpu_lib, *d, uneven_shards(V, 3, 2), beta, tau, keep)
    torch.testing.assert_close(rows3, ref_rows, rtol=1e-4, atol=1e-6)
    assert float(loss3.item()) == pytest.approx(float(ref.item()), rel=1e-4)


def test_fljsd_vp_identical_heads_is_zero(gpu_lib):
    T, H, V = 70, 128, 2000
    xs, Ws, _, _ = jsd_inputs(52, T, H, V, sw=0.2)
    xsd, Wsd = to_dev_bf16(xs), to_dev_bf16(Ws)
    _, _, terms, rows, loss = run_fljsd_vp(gpu_lib, xsd, Wsd, xsd, Wsd, uneven_shards(V, 3, 4), 0.5, 1.0)
    assert abs(float(loss.item())) <= 1e-6 and float(terms.abs().max()) <= 1e-6


def test_fljsd_vp_full_size_sampled(gpu_lib):
    """Student/teacher [1024, 4096], heads [128256, 4096] ~ N(0, 0.02^2) split
    over 4 ranks: the merged per-token JSD within 1e-4 of the unsharded call,
    sampled tokens against the oracle."""
    T, H, V, k = 1024, 4096, 128256, 4
    xs, Ws, xt, Wt = jsd_inputs(0, T, H, V, sw=0.02)
    d = [to_dev_bf16(a) for a in (xs, Ws, xt, Wt)]
    shards = [(j * V // k, (j + 1) * V // k - j * V // k) for j in range(k)]
    _, _, _, rows, loss = run_fljsd_vp(gpu_lib, *d, shards, 0.5, 1.0)
    ws = gpu_lib.workspace(gpu_lib.fljsd_workspace_bytes(T, H, V))
    ref = gpu_lib.fljsd_fwd_bf16(*d, 0.5, ws=ws)
    torch.testing.assert_close(rows, gpu_lib.row_losses(ws, T), rtol=1e-4, atol=1e-6)
    assert float(loss.item()) == pytest.approx(float(ref.item()), rel=1e-4)
    idx = np.array([0, 127, 128, 511, 512, 1023])
    _, want = oracle.fljsd_bf16(xs[idx], Ws, xt[idx], Wt, 0.5)
    np.testing.assert_allclose(np64(rows)[idx], want, rtol=RTOL_JSD_TOKEN, atol=ATOL_JSD_TOKEN)


def run_fljsd_vp_bwd(lmho, d, shards, beta, tau, keep, scale):
    """The vocab-parallel fused JSD forward and student backward over emulated
    shards: returns (lse [2, T], terms and KL shares [k, 2, T], KL [T], rows,
    loss, [(dxs share, dWs rows)])."""
    xsd, Wsd, xtd, Wtd = d
    T = xsd.shape[0]
    k = len(shards)
    local = [(Wsd[v0:v0 + w].clone(), Wtd[v0:v0 + w].clone()) for v0, w in shards]
    lparts = torch.full((k, 2, T), float("nan"), device="cuda")
    for j, (a, b) in enumerate(local):
        lmho.fljsd_lse_partials_bf16(xsd, a, xtd, b, tau, out=lparts[j])
    lse = lmho.lse_merge_partials(lparts)
    tk = torch.full((k, 2, T), float("nan"), device="cuda")
    for j, (a, b) in enumerate(local):
        lmho.fljsd_terms_bf16(xsd, a, xtd, b, lse, beta, tau, out=tk[j, 0], kl_local=tk[j, 1])
    loss, rows = lmho.jsd_merge_terms(tk[:, 0].contiguous(), keep)
    _, kl = lmho.jsd_merge_terms(tk[:, 1].contiguous())
    outs = [lmho.fljsd_shard_bwd_bf16(xsd, a, xtd, b, lse, kl, beta, tau, keep, scale) for a, b in local]
    torch.cuda.synchronize()
    return lse, tk, kl, rows, loss, outs


@pytest.mark.parametrize("T,H,V,k,beta,tau,masked", [(130, 128, 1000, 3, 0.5, 1.0, False),
                                                     (64, 256, 513, 2, 0.3, 2.0, True),
                                                     (96, 1024, 2000, 3, 0.5, 1.0, False),
                                                     (5, 64, 37, 4, 0.7, 0.8, True)])
def test_fljsd_vp_backward_matches_oracle(gpu_lib, T, H, V, k, beta, tau, masked):
    """KL shares against the oracle's; every shard's dxs share and dWs rows
    within their per-element bounds of the oracle's shard gradient; the
    shares' sum within the summed bounds of the unsharded oracle dxs."""
    xs, Ws, xt, Wt = jsd_inputs(80 + k, T, H, V, sw=2.0 / math.sqrt(H))
    keep = (np.arange(T) % 4 != 1).astype(np.uint8) if masked else None
    shards = uneven_shards(V, k, 20 + k)
    d = [to_dev_bf16(a) for a in (xs, Ws, xt, Wt)]
    _, tk, _, rows, loss, outs = run_fljsd_vp_bwd(gpu_lib, d, shards, beta, tau,
                                                  None if keep is None else to_dev(keep), 2.5)
    sl = [(np.ascontiguousarray(Ws[v0:v0 + w]), np.ascontiguousarray(Wt[v0:v0 + w])) for v0, w in shards]
    lse = oracle.lse_merge(np.stack([oracle.fljsd_lse_shard_bf16(xs, a, xt, b, tau) for a, b in sl]))
    kls = [oracle.fljsd_kl_shard_bf16(xs, a, xt, b, lse, beta, tau) for a, b in sl]
    kl = sum(kls)
    want_mean, want_rows = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, beta, tau, keep)
    np.testing.assert_allclose(np64(rows), want_rows, rtol=RTOL_JSD_TOKEN, atol=ATOL_JSD_TOKEN)
    assert float(loss.item()) == pytest.approx(want_mean, rel=RTOL_SCALAR)
    dz, gbp = oracle.fljsd_dz_bf16(xs, Ws, xt, Wt, beta, tau, keep, 2.5)
    xsd = gen.bf16_bits_to_f32(xs).astype(np.float64)
    Wsd = gen.bf16_bits_to_f32(Ws).astype(np.float64)
    dx_sum, b_sum = np.zeros((T, H)), np.zeros((T, H))
    for j, ((v0, w), (a, b)) in enumerate(zip(shards, sl)):
        np.testing.assert_allclose(np64(tk[j, 1]), kls[j], rtol=RTOL_JSD_TOKEN, atol=ATOL_JSD_TOKEN)
        bdx, bdW = grad_bounds(dz[:, v0:v0 + w], gbp[:, v0:v0 + w], xsd, Wsd[v0:v0 + w])
        dx_ref, dW_ref = oracle.fljsd_grad_shard_bf16(xs, a, xt, b, lse, kl, beta, tau, keep, 2.5)
        got_dx, got_dW = np64(outs[j][0]), np64(outs[j][1])
        assert_within_bounds(got_dx, dx_ref, bdx, f"dxs share of shard {j}")
        assert_within_bounds(got_dW, dW_ref, bdW, f"dWs rows of shard {j}")
        if masked:
            assert np.all(got_dx[keep == 0] == 0.0)
        dx_sum += got_dx
        b_sum += bdx
    dx_full, _ = oracle.fljsd_grad_bf16(xs, Ws, xt, Wt, beta, tau, keep, 2.5)
    assert_within_bounds(dx_sum, dx_full, b_sum, "sum of the dxs shares")


@pytest.mark.parametrize("masked", [False, True])
def test_fljsd_vp_backward_single_shard_bitwise(gpu_lib, masked):
    """One shard holding both whole heads: the loss and the student's dxs and
    dWs equal fljsd_fwd_bwd_bf16's bit for bit."""
    T, H, V = 200, 256, 3000
    xs, Ws, xt, Wt = jsd_inputs(85, T, H, V, sw=0.2)
    d = [to_dev_bf16(a) for a in (xs, Ws, xt, Wt)]
    keep = to_dev((np.arange(T) % 3 != 2).astype(np.uint8)) if masked else None
    ws = gpu_lib.workspace(gpu_lib.fljsd_bwd_workspace_bytes(T, H, V))
    ref_loss, ref_dx, ref_dW = gpu_lib.fljsd_fwd_bwd_bf16(*d, 0.4, 1.3, keep, 0.6, ws=ws)
    _, _, _, _, loss, outs = run_fljsd_vp_bwd(gpu_lib, d, [(0, V)], 0.4, 1.3, keep, 0.6)
    assert torch.equal(loss, ref_loss)
    assert torch.equal(outs[0][0], ref_dx) and torch.equal(outs[0][1], ref_dW)


# ---------------------------------------------------------------- CPO on the vocab-parallel fused CE
def run_cpo_vp(lmho, xd, Wd, td, shards, V, B, beta, alpha, scale):
    """Returns (loss, logps, row weights, [(dx share, dW rows)])."""
    parts, rows, _ = run_flce_vp(lmho, xd, Wd, td, shards, V)
    row_w = torch.full_like(rows, float("nan"))
    loss, logps = lmho.cpo_combine_rows(rows, B, beta, alpha, row_w=row_w)
    outs = [lmho.flce_shard_bwd_bf16(xd, Wd[v0:v0 + w].clone(), td, parts, v0, V, scale, row_w=row_w)
            for v0, w in shards]
    torch.cuda.synchronize()
    return loss, logps, row_w, outs


@pytest.mark.parametrize("B,S,H,V,k", [(4, 33, 128, 1000, 3), (2, 65, 256, 777, 2)])
def test_cpo_vp_matches_oracle(gpu_lib, B, S, H, V, k):
    """The CPO loss of the merged per-token losses against the oracle (2e-3),
    its weights against the oracle's combination of the oracle's losses, and
    every shard's weighted dx share and dW rows within their per-element
    bounds; the shares' sum within the summed bounds of the oracle's dx."""
    T = B * S
    x, W, t = flce_inputs(90 + k, T, H, V)
    shards = uneven_shards(V, k, 30 + k)
    loss, logps, row_w, outs = run_cpo_vp(gpu_lib, to_dev_bf16(x), to_dev_bf16(W), to_dev(t), shards, V, B, 0.3,
                                          0.7, 1.5)
    want, rows_ref, want_lp = oracle.cpo_bf16(x.reshape(B, S, H), W, t.reshape(B, S), 0.3, 0.7)
    assert float(loss.item()) == pytest.approx(want, rel=RTOL_SCALAR)
    np.testing.assert_allclose(np64(logps), want_lp, rtol=1e-4)
    _, _, w_ref = oracle.cpo_combine(rows_ref, 0.3, 0.7)
    np.testing.assert_allclose(np64(row_w), w_ref.reshape(T), rtol=1e-3, atol=1e-7)
    g = 1.5 * w_ref.reshape(T)
    dz = oracle.ce_grad_f64(oracle.logits_bf16(x, W), t, g, 1.0)
    S_err = ce_error_scale(dz, t, g)
    xd = gen.bf16_bits_to_f32(x).astype(np.float64)
    Wd = gen.bf16_bits_to_f32(W).astype(np.float64)
    dx_sum, b_sum = np.zeros((T, H)), np.zeros((T, H))
    for j, (v0, w) in enumerate(shards):
        bdx, bdW = grad_bounds(dz[:, v0:v0 + w], S_err[:, v0:v0 + w], xd, Wd[v0:v0 + w])
        # the weights themselves are fp32 values of the CPO combination: 1e-3 of each element's magnitude more
        got_dx, got_dW = np64(outs[j][0]), np64(outs[j][1])
        ref_dx, ref_dW = dz[:, v0:v0 + w] @ Wd[v0:v0 + w], dz[:, v0:v0 + w].T @ xd
        assert_within_bounds(got_dx, ref_dx, bdx + 1e-3 * np.abs(dz[:, v0:v0 + w]) @ np.abs(Wd[v0:v0 + w]),
                             f"dx share of shard {j}")
        assert_within_bounds(got_dW, ref_dW, bdW + 1e-3 * np.abs(dz[:, v0:v0 + w]).T @ np.abs(xd),
                             f"dW rows of shard {j}")
        dx_sum += got_dx
        b_sum += bdx + 1e-3 * np.abs(dz[:, v0:v0 + w]) @ np.abs(Wd[v0:v0 + w])
    dx_full, _ = oracle.cpo_grad_bf16(x.reshape(B, S, H), W, t.reshape(B, S), 0.3, 0.7, 1.5)
    assert_within_bounds(dx_sum, dx_full.reshape(T, H), b_sum, "sum of the dx shares")


def test_cpo_vp_single_shard_is_bitwise_flce_cpo(gpu_lib):
    """One shard holding all of W: the CPO loss, sequence log-likelihoods and
    gradients equal flce_cpo_fwd_bwd_bf16's bit for bit."""
    B, S, H, V = 4, 40, 256, 3000
    T = B * S
    x, W, t = flce_inputs(95, T, H, V)
    xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
    ws = gpu_lib.workspace(gpu_lib.flce_cpo_bwd_workspace_bytes(B, S, H, V))
    ref_loss, ref_lp, ref_dx, ref_dW = gpu_lib.flce_cpo_fwd_bwd_bf16(xd.view(B, S, H), Wd, td.view(B, S), 0.2, 0.5,
                                                                      1.3, ws=ws)
    loss, logps, _, outs = run_cpo_vp(gpu_lib, xd, Wd, td, [(0, V)], V, B, 0.2, 0.5, 1.3)
    assert torch.equal(loss, ref_loss) and torch.equal(logps, ref_lp)
    assert torch.equal(outs[0][0], ref_dx.view(T, H)) and torch.equal(outs[0][1], ref_dW)


# ---------------------------------------------------------------- merges alone
def test_lse_merge_and_rows_mean(gpu_lib):
    rng = np.random.default_rng(3)
    parts = rng.normal(0.0, 4.0, (3, 2, 1001)).astype(np.float32)
    got = np64(gpu_lib.lse_merge_partials(torch.from_numpy(parts).cuda()))
    want = np.logaddexp(np.logaddexp(parts[0].astype(np.float64), parts[1]), parts[2])
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-6)
    rows = torch.from_numpy(rng.normal(1.0, 1.0, 1003).astype(np.float32)).cuda()
    keep = torch.from_numpy((np.arange(1003) % 5 != 0).astype(np.uint8)).cuda()
    r = rows.double().cpu().numpy()
    assert float(gpu_lib.rows_mean(rows).item()) == pytest.approx(r.mean(), rel=1e-6)
    kk = keep.cpu().numpy() != 0
    assert float(gpu_lib.rows_mean(rows, keep).item()) == pytest.approx(r[kk].mean(), rel=1e-6)
    assert float(gpu_lib.rows_mean(rows, torch.zeros_like(keep)).item()) == 0.0


# ---------------------------------------------------------------- through dist.py and NCCL
def _nccl_one_rank(port, q):
    """Child process: a one-rank NCCL group runs the product helpers; with one
    rank the shard is the whole head, so they must give the unsharded calls'
    bits (the all-gathers and merges of one block are exact)."""
    import os

    import torch.distributed as dist

    import lm_head_online_gb300 as lmho
    from lm_head_online_gb300 import dist as lmdist

    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        torch.cuda.set_device(0)
        dist.init_process_group("nccl", rank=0, world_size=1)
        T, H, V = 256, 128, 2500
        x, W, t = flce_inputs(61, T, H, V)
        xd, Wd, td = to_dev_bf16(x), to_dev_bf16(W), to_dev(t)
        mean, rows = lmdist.vocab_parallel_flce(xd, Wd, td, 0, V)
        ws = lmho.workspace(lmho.flce_workspace_bytes(T, H, V))
        ref = lmho.flce_fwd_bf16(xd, Wd, td, ws=ws)
        ok_ce = torch.equal(rows, lmho.row_losses(ws, T)) and torch.equal(mean, ref)
        m2, rows2, dx, dW = lmdist.vocab_parallel_flce_fwd_bwd(xd, Wd, td, 0, V, 0.9)
        wsb = lmho.workspace(lmho.flce_bwd_workspace_bytes(T, H, V))
        ref_l, ref_dx, ref_dW = lmho.flce_fwd_bwd_bf16(xd, Wd, td, 0.9, ws=wsb)
        ok_ce = ok_ce and torch.equal(m2, ref_l) and torch.equal(dx, ref_dx) and torch.equal(dW, ref_dW)
        Bc, Sc = 4, T // 4
        l4, lp4, dx4, dW4 = lmdist.vocab_parallel_flce_cpo(xd, Wd, td, 0, V, Bc, 0.2, 0.6, backward=True,
                                                           grad_scale=1.1)
        wsc = lmho.workspace(lmho.flce_cpo_bwd_workspace_bytes(Bc, Sc, H, V))
        r4 = lmho.flce_cpo_fwd_bwd_bf16(xd.view(Bc, Sc, H), Wd, td.view(Bc, Sc), 0.2, 0.6, 1.1, ws=wsc)
        ok_ce = ok_ce and torch.equal(l4, r4[0]) and torch.equal(lp4, r4[1]) and torch.equal(dx4, r4[2].view(T, H)) \
            and torch.equal(dW4, r4[3])
        xs, Ws, xt, Wt = jsd_inputs(62, T, H, V, sw=0.2)
        d = [to_dev_bf16(a) for a in (xs, Ws, xt, Wt)]
        keep = to_dev((np.arange(T) % 5 != 3).astype(np.uint8))
        loss, jrows = lmdist.vocab_parallel_fljsd(*d, 0.4, 1.5, keep)
        ws2 = lmho.workspace(lmho.fljsd_workspace_bytes(T, H, V))
        ref2 = lmho.fljsd_fwd_bf16_ex(*d, 0.4, 1.5, keep, ws=ws2)
        ok_jsd = torch.equal(jrows, lmho.row_losses(ws2, T)) and torch.equal(loss, ref2)
        l3, r3, dxs, dWs = lmdist.vocab_parallel_fljsd_fwd_bwd(*d, 0.4, 1.5, keep, 0.8)
        ws3 = lmho.workspace(lmho.fljsd_bwd_workspace_bytes(T, H, V))
        ref3, ref_dxs, ref_dWs = lmho.fljsd_fwd_bwd_bf16(*d, 0.4, 1.5, keep, 0.8, ws=ws3)
        ok_jsd = ok_jsd and torch.equal(l3, ref3) and torch.equal(dxs, ref_dxs) and torch.equal(dWs, ref_dWs)
        dist.destroy_process_group()
        q.put((ok_ce, ok_jsd, None))
    except Exception as e:  # report to the parent
        q.put((False, False, repr(e)))


def test_vocab_parallel_helpers_over_nccl_one_rank(gpu_lib):
    import socket

    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_nccl_one_rank, args=(port, q))
    p.start()
    ok_ce, ok_jsd, err = q.get(timeout=300)
    p.join(timeout=60)
    assert err is None, err
    assert ok_ce and ok_jsd
    assert p.exitcode == 0
