"""Pins of the vocab-parallel cross-entropy oracle (page "Vocab-parallel
cross-entropy, Megatron layout", summary: the vocabulary is split across
tensor-parallel ranks, so each rank holds logits [seq, batch, V_local] of its
own vocab range).  Each shard reduces a row to (max, sum of exp, target logit or
-inf); the shards' triples combine into the row's loss.

The pins check the oracle against things other than itself: a 40-digit
brute force of the per-shard sums, the unsharded Megatron-layout oracle
(itself pinned in test_oracle_ce.py) for every split, closed forms, the
ownership of targets on shard edges and the independence of the result from
the order of the shards."""
import math

import mpmath
import numpy as np
import pytest

import gen
import oracle


def bits_of(vals):
    """bf16 bit patterns of values exactly representable in bf16."""
    f = np.asarray(vals, np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


def splits(V, k, seed):
    """k shard widths >= 1 summing to V, uneven."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, V), size=k - 1, replace=False)) if k > 1 else np.array([], int)
    edges = np.concatenate([[0], cuts, [V]])
    return [(int(a), int(b - a)) for a, b in zip(edges[:-1], edges[1:])]


def shard_partials(z, t, shards):
    parts = [oracle.ce_partials_bf16(np.ascontiguousarray(z[..., v0:v0 + w]), t, v0) for v0, w in shards]
    return tuple(np.stack([p[i] for p in parts]) for i in range(3))


def test_partials_brute_force_40_digits():
    vals = np.array([[1.5, -2.0, 0.25, 3.0, -7.5], [0.0, 0.0, 0.0, -0.5, 2.5]], np.float32)
    z = bits_of(vals)
    t = np.array([3, 0])
    m, s, zt = oracle.ce_partials_bf16(z, t, v0=0)
    mpmath.mp.dps = 40
    for r in range(2):
        row = [mpmath.mpf(float(x)) for x in vals[r]]
        M = max(row)
        S = mpmath.fsum(mpmath.exp(x - M) for x in row)
        assert m[r] == float(M)
        assert s[r] == pytest.approx(float(S), rel=1e-15)
        assert zt[r] == float(vals[r, t[r]])


def test_target_ownership_and_edges():
    V, rows = 37, 6
    z = gen.normal_bf16_bits(5, 0, (rows, V), sigma=2.0)
    shards = [(0, 10), (10, 1), (11, 20), (31, 6)]
    for v0, w in shards:
        for t_val in (v0, v0 + w - 1, v0 - 1, v0 + w, -1, V):
            t = np.full(rows, t_val)
            _, _, zt = oracle.ce_partials_bf16(np.ascontiguousarray(z[:, v0:v0 + w]), t, v0)
            if v0 <= t_val < v0 + w:
                want = (z[:, t_val].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                np.testing.assert_array_equal(zt, want)
            else:
                assert np.all(zt == -np.inf)


@pytest.mark.parametrize("k", [1, 2, 3, 7])
def test_merge_equals_unsharded(k):
    S, B, V = 5, 3, 1001
    z = gen.normal_bf16_bits(6, 0, (S, B, V), sigma=2.0)
    t = gen.targets(6, 1, (S, B), V)
    shards = splits(V, k, seed=k)
    got = oracle.ce_merge(*shard_partials(z, t, shards), t, V)
    want = oracle.ce_sbv_bf16(z, t)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_merge_targets_on_shard_edges():
    S, B, V = 4, 4, 64
    z = gen.normal_bf16_bits(7, 0, (S, B, V), sigma=3.0)
    shards = [(0, 5), (5, 1), (6, 33), (39, 25)]
    edges = [v for v0, w in shards for v in (v0, v0 + w - 1)]
    t = np.array(edges * 4)[: S * B].reshape(S, B)
    got = oracle.ce_merge(*shard_partials(z, t, shards), t, V)
    np.testing.assert_allclose(got, oracle.ce_sbv_bf16(z, t), rtol=1e-12, atol=1e-12)


def test_merge_order_of_shards():
    S, B, V = 3, 2, 300
    z = gen.normal_bf16_bits(8, 0, (S, B, V), sigma=2.0)
    t = gen.targets(8, 1, (S, B), V)
    shards = splits(V, 5, seed=3)
    m, s, zt = shard_partials(z, t, shards)
    a = oracle.ce_merge(m, s, zt, t, V)
    perm = [3, 0, 4, 2, 1]
    b = oracle.ce_merge(m[perm], s[perm], zt[perm], t, V)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


def test_equal_logits_give_ln_V():
    S, B, V = 2, 2, 96
    z = np.full((S, B, V), bits_of([1.25])[0], np.uint16)
    t = np.array([[0, 95], [40, 41]])
    got = oracle.ce_merge(*shard_partials(z, t, [(0, 7), (7, 50), (57, 39)]), t, V)
    np.testing.assert_allclose(got, np.full((S, B), math.log(V)), rtol=0, atol=1e-14)


def test_out_of_range_target_is_nan_and_single_shard_is_plain_ce():
    S, B, V = 2, 3, 50
    z = gen.normal_bf16_bits(9, 0, (S, B, V), sigma=2.0)
    t = gen.targets(9, 1, (S, B), V)
    t[0, 1], t[1, 2] = -1, V
    m, s, zt = oracle.ce_partials_bf16(z, t, 0)
    loss = oracle.ce_merge(m[None], s[None], zt[None], t, V)
    assert math.isnan(loss[0, 1]) and math.isnan(loss[1, 2])
    ok = np.ones((S, B), bool)
    ok[0, 1] = ok[1, 2] = False
    np.testing.assert_allclose(loss[ok], oracle.ce_sbv_bf16(z, t)[ok], rtol=1e-13)
    # one shard: m + ln s - zt is the plain cross-entropy of the row
    np.testing.assert_allclose((m + np.log(s) - zt)[ok], oracle.ce_sbv_bf16(z, t)[ok], rtol=1e-13)


@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_flat_f32_shards_merge_to_unsharded(k):
    """The flat fp32 layout's shard partials (the cross-entropy page's
    [tokens, vocab] logits with the vocab split the same way) merge into the
    unsharded flat oracle's per-token losses, targets on shard edges."""
    T, V = 9, 233
    z = gen.normal_f32(12, 0, (T, V))
    t = gen.targets(12, 1, (T,), V)
    shards = splits(V, k, 30 + k)
    edge = [c for v0, w in shards for c in (v0, v0 + w - 1)]
    t[:min(T, len(edge))] = edge[:T]
    parts = [oracle.ce_partials_f32(np.ascontiguousarray(z[:, v0:v0 + w]), t, v0) for v0, w in shards]
    m, s, zt = (np.stack([p[i] for p in parts]) for i in range(3))
    _, want = oracle.ce_f32(z, t)
    np.testing.assert_allclose(oracle.ce_merge(m, s, zt, t, V), want, rtol=1e-12, atol=1e-12)
