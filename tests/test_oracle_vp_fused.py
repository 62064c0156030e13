"""Pins of the oracle's vocab-parallel fused losses: the vocabulary split of
the page "Vocab-parallel cross-entropy, Megatron layout" (summary: each
tensor-parallel rank holds its own vocab range) applied to the output layer,
so a rank holds the rows [v0, v0 + V_local) of W and its logits are
x W_local^T.

  * fused CE: each shard reduces its logits to (max, sum of exp, target logit
    or -inf); the triples combine into the loss as for the Megatron layout.
  * fused JSD (page "Fused linear + JSD"): each shard gives each head's
    log-sum-exp over its columns; these combine into the global ones; with
    them each shard sums its columns' JSD terms, and the sums combine into the
    per-token JSD and its batchmean.

The pins check these against things other than themselves: the unsharded
fused oracles (pinned in test_oracle_fused.py) for every split, scipy's
logsumexp and numpy's logaddexp, closed forms (x = 0, identical heads) and
hand-computed merges."""
import math

import numpy as np
import pytest
import scipy.special as sp

import gen
import oracle


def splits(V, k, seed):
    """k shard widths >= 1 summing to V, uneven."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, V), size=k - 1, replace=False)) if k > 1 else np.array([], int)
    edges = np.concatenate([[0], cuts, [V]])
    return [(int(a), int(b - a)) for a, b in zip(edges[:-1], edges[1:])]


def flce_inputs(seed, T, H, V):
    x = gen.normal_bf16_bits(seed, 0, (T, H), sigma=1.0)
    W = gen.normal_bf16_bits(seed, 1, (V, H), sigma=0.3)
    t = gen.targets(seed, 2, (T,), V)
    return x, W, t


def jsd_inputs(seed, T, H, V):
    xs = gen.normal_bf16_bits(seed, 0, (T, H), sigma=1.0)
    Ws = gen.normal_bf16_bits(seed, 1, (V, H), sigma=0.3)
    xt = gen.normal_bf16_bits(seed, 2, (T, H), sigma=1.0)
    Wt = gen.normal_bf16_bits(seed, 3, (V, H), sigma=0.3)
    return xs, Ws, xt, Wt


def flce_partials(x, W, t, shards):
    parts = [oracle.flce_partials_bf16(x, np.ascontiguousarray(W[v0:v0 + w]), t, v0) for v0, w in shards]
    return tuple(np.stack([p[i] for p in parts]) for i in range(3))


@pytest.mark.parametrize("k", [1, 2, 3, 5])
def test_flce_shards_merge_to_unsharded(k):
    T, H, V = 9, 24, 61
    x, W, t = flce_inputs(7 + k, T, H, V)
    shards = splits(V, k, 11 + k)
    # targets on every shard's first and last column
    edge = [c for v0, w in shards for c in (v0, v0 + w - 1)]
    t[:len(edge[:T])] = edge[:T]
    m, s, zt = flce_partials(x, W, t, shards)
    got = oracle.ce_merge(m, s, zt, t, V)
    _, want = oracle.flce_bf16(x, W, t)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_flce_partials_own_their_targets():
    T, H, V = 6, 16, 40
    x, W, t = flce_inputs(3, T, H, V)
    t[:] = [0, 9, 10, 25, 39, 17]
    shards = [(0, 10), (10, 16), (26, 14)]
    _, _, zt = flce_partials(x, W, t, shards)
    z = oracle.logits_bf16(x, W)
    for j, (v0, w) in enumerate(shards):
        for i in range(T):
            if v0 <= t[i] < v0 + w:
                assert zt[j, i] == z[i, t[i]]
            else:
                assert zt[j, i] == -math.inf
    # each target is owned by exactly one shard
    assert np.all(np.isfinite(zt).sum(axis=0) == 1)


def test_flce_partials_x_zero_closed_form():
    """x = 0: every logit is 0, so a shard of width w has m = 0 and s = w, and
    the merged loss is ln V."""
    T, H, V = 4, 16, 50
    x = np.zeros((T, H), np.uint16)
    _, W, t = flce_inputs(5, T, H, V)
    shards = splits(V, 3, 2)
    m, s, zt = flce_partials(x, W, t, shards)
    assert np.all(m == 0.0)
    np.testing.assert_array_equal(s, np.array([[w] * T for _, w in shards], np.float64))
    np.testing.assert_allclose(oracle.ce_merge(m, s, zt, t, V), math.log(V), rtol=1e-15)


def test_flce_out_of_range_target_is_nan():
    T, H, V = 3, 16, 30
    x, W, t = flce_inputs(9, T, H, V)
    t[:] = [-1, V, 4]
    m, s, zt = flce_partials(x, W, t, splits(V, 2, 1))
    loss = oracle.ce_merge(m, s, zt, t, V)
    assert math.isnan(loss[0]) and math.isnan(loss[1]) and math.isfinite(loss[2])


@pytest.mark.parametrize("tau", [1.0, 0.7, 2.0])
def test_fljsd_lse_shard_is_scipy_logsumexp(tau):
    T, H, V = 5, 24, 47
    xs, Ws, xt, Wt = jsd_inputs(13, T, H, V)
    zs, zq = oracle.logits_bf16(xs, Ws), oracle.logits_bf16(xt, Wt)
    for v0, w in splits(V, 3, 4):
        got = oracle.fljsd_lse_shard_bf16(xs, np.ascontiguousarray(Ws[v0:v0 + w]), xt,
                                          np.ascontiguousarray(Wt[v0:v0 + w]), tau)
        np.testing.assert_allclose(got[0], sp.logsumexp(zs[:, v0:v0 + w] / tau, axis=1), rtol=1e-13)
        np.testing.assert_allclose(got[1], sp.logsumexp(zq[:, v0:v0 + w] / tau, axis=1), rtol=1e-13)


def test_lse_merge_is_logaddexp():
    rng = np.random.default_rng(0)
    parts = rng.normal(0.0, 5.0, (3, 2, 11))
    parts[1, 0, 3] = 700.0   # a large value: the max-shifted form does not overflow
    want = np.logaddexp(np.logaddexp(parts[0], parts[1]), parts[2])
    np.testing.assert_allclose(oracle.lse_merge(parts), want, rtol=1e-14)
    np.testing.assert_array_equal(oracle.lse_merge(parts[:1]), parts[0])


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("beta,tau,masked", [(0.5, 1.0, False), (0.3, 2.0, True), (0.8, 0.7, False)])
def test_fljsd_shards_merge_to_unsharded(k, beta, tau, masked):
    T, H, V = 8, 24, 53
    xs, Ws, xt, Wt = jsd_inputs(17 + k, T, H, V)
    keep = (np.arange(T) % 3 != 1).astype(np.uint8) if masked else None
    shards = splits(V, k, 5 + k)
    sl = [(np.ascontiguousarray(Ws[v0:v0 + w]), np.ascontiguousarray(Wt[v0:v0 + w])) for v0, w in shards]
    lse = oracle.lse_merge(np.stack([oracle.fljsd_lse_shard_bf16(xs, a, xt, b, tau) for a, b in sl]))
    terms = np.stack([oracle.fljsd_terms_shard_bf16(xs, a, xt, b, lse, beta, tau) for a, b in sl])
    mean, rows = oracle.jsd_merge(terms, keep)
    want_mean, want_rows = oracle.fljsd_ex_bf16(xs, Ws, xt, Wt, beta, tau, keep)
    np.testing.assert_allclose(rows, want_rows, rtol=1e-11, atol=1e-15)
    assert mean == pytest.approx(want_mean, rel=1e-11)


def test_fljsd_identical_heads_give_zero_terms():
    T, H, V = 4, 16, 33
    xs, Ws, _, _ = jsd_inputs(21, T, H, V)
    shards = splits(V, 3, 3)
    sl = [np.ascontiguousarray(Ws[v0:v0 + w]) for v0, w in shards]
    lse = oracle.lse_merge(np.stack([oracle.fljsd_lse_shard_bf16(xs, a, xs, a) for a in sl]))
    for a in sl:
        assert np.abs(oracle.fljsd_terms_shard_bf16(xs, a, xs, a, lse)).max() <= 1e-15


def test_jsd_merge_by_hand():
    terms = np.array([[1.0, 2.0, 0.5], [3.0, 4.0, 0.25]])
    mean, rows = oracle.jsd_merge(terms)
    np.testing.assert_array_equal(rows, [4.0, 6.0, 0.75])
    assert mean == pytest.approx((4.0 + 6.0 + 0.75) / 3, rel=1e-15)
    mean, rows = oracle.jsd_merge(terms, np.array([1, 0, 1], np.uint8))
    np.testing.assert_array_equal(rows, [4.0, 0.0, 0.75])
    assert mean == pytest.approx(4.75 / 2, rel=1e-15)
    mean, rows = oracle.jsd_merge(terms, np.zeros(3, np.uint8))
    assert mean == 0.0 and np.all(rows == 0.0)


# ---------------------------------------------------------------- fused CE backward of a shard
def test_partials_lse_is_scipy_logsumexp():
    T, H, V = 7, 24, 59
    x, W, t = flce_inputs(41, T, H, V)
    m, s, _ = flce_partials(x, W, t, splits(V, 3, 8))
    np.testing.assert_allclose(oracle.ce_partials_lse(m, s), sp.logsumexp(oracle.logits_bf16(x, W), axis=1),
                               rtol=1e-14)


@pytest.mark.parametrize("k", [1, 2, 3])
def test_flce_shard_grads_sum_to_unsharded(k):
    """The shards' dx shares add up to the unsharded dx and their dW rows stack
    into the unsharded dW (targets on shard edges, scale 1.7)."""
    T, H, V = 6, 16, 47
    x, W, t = flce_inputs(43 + k, T, H, V)
    shards = splits(V, k, 2 + k)
    edge = [c for v0, w in shards for c in (v0, v0 + w - 1)]
    t[:min(T, len(edge))] = edge[:T]
    m, s, _ = flce_partials(x, W, t, shards)
    lse = oracle.ce_partials_lse(m, s)
    dx_full, dW_full = oracle.flce_grad_bf16(x, W, t, 1.7)
    dx_sum = np.zeros_like(dx_full)
    for v0, w in shards:
        dx, dW = oracle.flce_grad_shard_bf16(x, np.ascontiguousarray(W[v0:v0 + w]), t, v0, V, lse, 1.7)
        dx_sum += dx
        np.testing.assert_allclose(dW, dW_full[v0:v0 + w], rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(dx_sum, dx_full, rtol=1e-11, atol=1e-15)


def test_flce_shard_grad_bad_target_is_nan_row():
    T, H, V = 4, 16, 30
    x, W, t = flce_inputs(47, T, H, V)
    t[1] = V
    m, s, _ = flce_partials(x, W, t, [(0, 12), (12, 18)])
    dx, dW = oracle.flce_grad_shard_bf16(x, np.ascontiguousarray(W[:12]), t, 0, V, oracle.ce_partials_lse(m, s))
    assert np.all(np.isnan(dx[1])) and np.all(np.isfinite(np.delete(dx, 1, axis=0))) and np.all(np.isnan(dW))


# ---------------------------------------------------------------- fused JSD student backward of a shard
def _jsd_shard_setup(seed, T, H, V, k, tau):
    xs, Ws, xt, Wt = jsd_inputs(seed, T, H, V)
    shards = splits(V, k, seed)
    sl = [(np.ascontiguousarray(Ws[v0:v0 + w]), np.ascontiguousarray(Wt[v0:v0 + w])) for v0, w in shards]
    lse = oracle.lse_merge(np.stack([oracle.fljsd_lse_shard_bf16(xs, a, xt, b, tau) for a, b in sl]))
    return xs, Ws, xt, Wt, shards, sl, lse


@pytest.mark.parametrize("beta,tau", [(0.5, 1.0), (0.3, 1.7)])
def test_fljsd_kl_shares_sum_to_scipy_rel_entr(beta, tau):
    T, H, V = 6, 16, 43
    xs, Ws, xt, Wt, shards, sl, lse = _jsd_shard_setup(51, T, H, V, 3, tau)
    kl = sum(oracle.fljsd_kl_shard_bf16(xs, a, xt, b, lse, beta, tau) for a, b in sl)
    P = sp.softmax(oracle.logits_bf16(xs, Ws) / tau, axis=1)
    Q = sp.softmax(oracle.logits_bf16(xt, Wt) / tau, axis=1)
    np.testing.assert_allclose(kl, sp.rel_entr(P, beta * P + (1 - beta) * Q).sum(axis=1), rtol=1e-11, atol=1e-15)


@pytest.mark.parametrize("k", [1, 2, 3])
@pytest.mark.parametrize("beta,tau,masked", [(0.5, 1.0, False), (0.3, 2.0, True)])
def test_fljsd_shard_grads_sum_to_unsharded(k, beta, tau, masked):
    T, H, V = 6, 16, 41
    xs, Ws, xt, Wt, shards, sl, lse = _jsd_shard_setup(53 + k, T, H, V, k, tau)
    keep = (np.arange(T) % 3 != 1).astype(np.uint8) if masked else None
    kl = sum(oracle.fljsd_kl_shard_bf16(xs, a, xt, b, lse, beta, tau) for a, b in sl)
    dx_full, dW_full = oracle.fljsd_grad_bf16(xs, Ws, xt, Wt, beta, tau, keep, 1.4)
    dx_sum = np.zeros_like(dx_full)
    for (v0, w), (a, b) in zip(shards, sl):
        dx, dW = oracle.fljsd_grad_shard_bf16(xs, a, xt, b, lse, kl, beta, tau, keep, 1.4)
        dx_sum += dx
        np.testing.assert_allclose(dW, dW_full[v0:v0 + w], rtol=1e-10, atol=1e-15)
        if masked:
            assert np.all(dx[keep == 0] == 0.0)
    np.testing.assert_allclose(dx_sum, dx_full, rtol=1e-10, atol=1e-15)
