"""GPU parity of the vocab-parallel (tensor-parallel) Megatron cross-entropy
against the fp64 oracle.

Page "Vocab-parallel cross-entropy, Megatron layout", summary: with the
vocabulary sharded over tensor-parallel ranks, each rank holds logits
[seq, batch, V_local] of its own vocab range.  Here the ranks are emulated on
one GPU: the global bf16 logits are cut into k uneven shards in device memory,
each shard's partials come from ce_partials_sbv_bf16, and ce_merge_partials
combines the k blocks (laid out as an all-gather in rank order would leave
them) into per-token losses.

Tolerances: partial maxima and target logits are bf16 values widened to fp32,
so they must be exact; partial sums of exp are fp32 sums of ex2.approx terms
with an online rescale: relative 1e-5.  Losses: the bf16 bar of absolute
2e-3 per token, and within 1e-5 relative (1e-6 absolute) of the single-GPU
ce_fwd_sbv_bf16 on the same logits.
"""
import math

import numpy as np
import pytest
import torch

import gen
import oracle
from tests.helpers import rows_bf16, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

ATOL_BF16 = 2e-3
RTOL_SUM = 1e-5


@pytest.fixture(autouse=True)
def _auto_variant(gpu_lib):
    gpu_lib.set_ce_variant("auto")
    yield
    gpu_lib.set_ce_variant("auto")


def uneven_shards(V, k, seed):
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, V), size=k - 1, replace=False))
    edges = np.concatenate([[0], cuts, [V]])
    return [(int(a), int(b - a)) for a, b in zip(edges[:-1], edges[1:])]


def run_vp(lmho, zd, td, shards, V):
    """zd: device bf16 [S, B, V]; each shard copied to its own contiguous
    buffer (a rank's local logits); returns (partials [k, 3, S, B], loss)."""
    S, B, _ = zd.shape
    parts = torch.full((len(shards), 3, S, B), float("nan"), device="cuda")
    for j, (v0, w) in enumerate(shards):
        local = zd[:, :, v0:v0 + w].contiguous()
        lmho.ce_partials_sbv_bf16(local, td, v0, partials=parts[j])
    loss = lmho.ce_merge_partials(parts, td, V)
    torch.cuda.synchronize()
    return parts, loss


def check_partials(parts, z, t, shards):
    got = parts.cpu().numpy().astype(np.float64)
    for j, (v0, w) in enumerate(shards):
        m, s, zt = oracle.ce_partials_bf16(np.ascontiguousarray(z[..., v0:v0 + w]), t, v0)
        np.testing.assert_array_equal(got[j, 0], m)
        np.testing.assert_allclose(got[j, 1], s, rtol=RTOL_SUM)
        np.testing.assert_array_equal(got[j, 2], zt)


SHAPES = [(1, 1, 7), (3, 2, 64), (7, 4, 1001), (16, 4, 4096), (5, 3, 20000)]


@pytest.mark.parametrize("k", [2, 3, 8])
@pytest.mark.parametrize("S,B,V", SHAPES)
def test_vocab_parallel_matches_oracle(gpu_lib, S, B, V, k):
    if V < k:
        pytest.skip("fewer columns than shards")
    z = gen.normal_bf16_bits(11, 0, (S, B, V), sigma=2.0)
    t = gen.targets(11, 1, (S, B), V)
    shards = uneven_shards(V, k, seed=V + k)
    zd, td = to_dev_bf16(z), to_dev(t)
    parts, loss = run_vp(gpu_lib, zd, td, shards, V)
    check_partials(parts, z, t, shards)
    ref = oracle.ce_sbv_bf16(z, t)
    got = loss.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=0, atol=ATOL_BF16)
    single = gpu_lib.ce_fwd_sbv_bf16(zd, td).cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got, single, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("variant", ["warp", "cta", "cta512", "cluster2", "cluster8", "bulk"])
def test_every_decomposition_and_shard_edges(gpu_lib, variant):
    """Targets on the first and last column of every shard, shards of width 1
    and odd widths (rows not 16-byte aligned: scalar heads and tails)."""
    gpu_lib.set_ce_variant(variant)
    S, B, V = 8, 4, 3001
    shards = [(0, 1), (1, 700), (701, 1), (702, 1299), (2001, 1000)]
    z = gen.normal_bf16_bits(12, 0, (S, B, V), sigma=2.0)
    edges = [v for v0, w in shards for v in (v0, v0 + w - 1)]
    t = np.array((edges * 4)[: S * B], np.int64).reshape(S, B)
    zd, td = to_dev_bf16(z), to_dev(t)
    parts, loss = run_vp(gpu_lib, zd, td, shards, V)
    check_partials(parts, z, t, shards)
    np.testing.assert_allclose(loss.cpu().numpy(), oracle.ce_sbv_bf16(z, t), rtol=0, atol=ATOL_BF16)


def test_out_of_range_targets_and_nan_logits(gpu_lib):
    S, B, V = 4, 2, 500
    shards = uneven_shards(V, 3, seed=1)
    z = gen.normal_bf16_bits(13, 0, (S, B, V), sigma=2.0)
    t = gen.targets(13, 1, (S, B), V)
    t[0, 0], t[1, 1] = -1, V          # no shard owns these
    z[2, 0, 77] = 0x7FC0              # a NaN logit in token (2, 0)
    parts, loss = run_vp(gpu_lib, to_dev_bf16(z), to_dev(t), shards, V)
    got = loss.cpu().numpy()
    assert math.isnan(got[0, 0]) and math.isnan(got[1, 1]) and math.isnan(got[2, 0])
    ok = np.ones((S, B), bool)
    ok[0, 0] = ok[1, 1] = ok[2, 0] = False
    np.testing.assert_allclose(got[ok], oracle.ce_sbv_bf16(z, t)[ok], rtol=0, atol=ATOL_BF16)
    # the shards that do not own a target hold -inf as its logit
    zt = parts[:, 2].cpu().numpy()
    owners = [sum(1 for v0, w in shards if v0 <= t[i, b] < v0 + w) for i in range(S) for b in range(B)]
    assert np.sum(np.isneginf(zt)) == len(shards) * S * B - sum(owners)


def test_one_shard_is_the_plain_megatron_loss(gpu_lib):
    S, B, V = 32, 4, 8192
    z = gen.normal_bf16_bits(14, 0, (S, B, V), sigma=2.0)
    t = gen.targets(14, 1, (S, B), V)
    zd, td = to_dev_bf16(z), to_dev(t)
    parts, loss = run_vp(gpu_lib, zd, td, [(0, V)], V)
    np.testing.assert_array_equal(loss.cpu().numpy(), gpu_lib.ce_fwd_sbv_bf16(zd, td).cpu().numpy())


def test_repeated_calls_bitwise_equal(gpu_lib):
    S, B, V = 64, 4, 12345
    shards = uneven_shards(V, 4, seed=2)
    z = gen.normal_bf16_bits(15, 0, (S, B, V), sigma=2.0)
    t = gen.targets(15, 1, (S, B), V)
    zd, td = to_dev_bf16(z), to_dev(t)
    first = run_vp(gpu_lib, zd, td, shards, V)[1].cpu().numpy()
    for _ in range(3):
        np.testing.assert_array_equal(run_vp(gpu_lib, zd, td, shards, V)[1].cpu().numpy(), first)


def test_full_size_eight_shards_sampled(gpu_lib):
    """The largest Megatron workload, bf16 [2048, 4, 131072] ~ N(0, 2^2), split
    into 8 equal shards of 16384 columns (tensor-parallel size 8): every
    token's loss against the single-GPU kernel, sampled tokens against the
    oracle on rows regenerated on the host."""
    S, B, V = 2048, 4, 131072
    z = torch.empty((S, B, V), dtype=torch.bfloat16)
    gen.normal_bf16_bits(0, 0, (S, B, V), 2.0, out=z.view(torch.int16))
    t = gen.targets(0, 1, (S, B), V)
    zd, td = z.cuda(), to_dev(t)
    del z
    shards = [(j * V // 8, V // 8) for j in range(8)]
    parts, loss = run_vp(gpu_lib, zd, td, shards, V)
    single = gpu_lib.ce_fwd_sbv_bf16(zd, td)
    np.testing.assert_allclose(loss.cpu().numpy(), single.cpu().numpy(), rtol=1e-5, atol=1e-6)
    idx = sample_rows(S * B, 32, seed=5)
    rows = rows_bf16(0, 0, idx, V, sigma=2.0)
    ref = oracle.ce_sbv_bf16(rows.reshape(-1, 1, V), t.reshape(-1)[idx].reshape(-1, 1)).reshape(-1)
    np.testing.assert_allclose(loss.cpu().numpy().reshape(-1)[idx], ref, rtol=0, atol=ATOL_BF16)


# ---------------------------------------------------------------- the flat fp32 layout
def run_vp_f32(lmho, zd, td, shards, V):
    """zd: device fp32 [T, V]; each shard copied to its own buffer; returns
    (partials [k, 3, T], per-token losses [T], mean [1])."""
    T = zd.shape[0]
    parts = torch.full((len(shards), 3, T), float("nan"), device="cuda")
    for j, (v0, w) in enumerate(shards):
        lmho.ce_partials_f32(zd[:, v0:v0 + w].contiguous(), td, v0, partials=parts[j])
    rows = lmho.ce_merge_partials(parts.view(len(shards), 3, T, 1), td.view(T, 1), V).view(T)
    mean = lmho.rows_mean(rows)
    torch.cuda.synchronize()
    return parts, rows, mean


@pytest.mark.parametrize("variant", ["auto", "warp", "cta", "cta512", "cluster2", "cluster8", "bulk"])
@pytest.mark.parametrize("T,V,k", [(37, 1001, 3), (130, 4099, 2), (5, 40000, 4)])
def test_flat_f32_vocab_parallel_matches_oracle(gpu_lib, variant, T, V, k):
    """Flat fp32 logits (page "Cross-entropy loss") with the vocabulary split:
    partial maxima and target logits exact (fp32 values), partial sums rel
    1e-5, per-token losses and the mean rel 1e-5 of the oracle (the flat bar);
    targets on the first and last column of every shard."""
    gpu_lib.set_ce_variant(variant)
    z = gen.normal_f32(16, 0, (T, V))
    t = gen.targets(16, 1, (T,), V)
    shards = uneven_shards(V, k, seed=T + k)
    edges = [c for v0, w in shards for c in (v0, v0 + w - 1)]
    t[:min(T, len(edges))] = edges[:T]
    parts, rows, mean = run_vp_f32(gpu_lib, to_dev(z), to_dev(t), shards, V)
    got = parts.cpu().numpy().astype(np.float64)
    for j, (v0, w) in enumerate(shards):
        m, s, zt = oracle.ce_partials_f32(np.ascontiguousarray(z[:, v0:v0 + w]), t, v0)
        np.testing.assert_array_equal(got[j, 0], m)
        np.testing.assert_allclose(got[j, 1], s, rtol=RTOL_SUM)
        np.testing.assert_array_equal(got[j, 2], zt)
    want_mean, want = oracle.ce_f32(z, t)
    np.testing.assert_allclose(rows.cpu().numpy().astype(np.float64), want, rtol=1e-5, atol=1e-6)
    assert float(mean.item()) == pytest.approx(want_mean, rel=1e-5)


def test_flat_f32_one_shard_is_ce_fwd_f32_bitwise(gpu_lib):
    T, V = 300, 4096
    z = gen.normal_f32(17, 0, (T, V))
    t = gen.targets(17, 1, (T,), V)
    zd, td = to_dev(z), to_dev(t)
    ws = gpu_lib.workspace(gpu_lib.ce_workspace_bytes(T, V))
    ref = gpu_lib.ce_fwd_f32(zd, td, ws=ws)
    _, rows, mean = run_vp_f32(gpu_lib, zd, td, [(0, V)], V)
    assert torch.equal(rows, gpu_lib.row_losses(ws, T)) and torch.equal(mean, ref)
