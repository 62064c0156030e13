"""Multi-process paths on CPU with the gloo backend, world size 2.

* Token sharding (what `bench.py --gpus N` runs): each rank takes a
  contiguous token slice; the per-rank means combine into the global mean.
* Vocab-parallel cross-entropy (page "Vocab-parallel cross-entropy, Megatron
  layout": vocab sharded over tensor-parallel ranks): each rank reduces its
  vocab shard to per-token (max, sum of exp, target logit or -inf),
  dist.gather_partials all-gathers them in rank order, and the merge gives
  the unsharded loss.  The ranks' reductions and the merge here are the
  oracle's (no GPU); the GPU kernels of the same steps are checked against
  the oracle in test_gpu_vp.py.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import gen
import oracle
from lm_head_online_gb300 import dist as lmdist


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(rank, world, port, fn, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, fn(rank, world)))
    except Exception as e:  # report failures to the parent
        q.put((rank, e))
    finally:
        dist.destroy_process_group()


def spawn(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_run, args=(r, world, port, fn, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, v in out.items():
        if isinstance(v, Exception):
            raise v
    return out


def test_shard_rows_cover_and_balance():
    for T in (1, 2, 7, 16384):
        for world in (1, 2, 3, 8):
            spans = [lmdist.shard_rows(T, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        lmdist.shard_rows(4, 2, 2)


def _token_sharded(rank, world):
    T, V = 37, 300
    z = gen.normal_f32(3, 0, (T, V))
    t = gen.targets(3, 1, (T,), V)
    lo, hi = lmdist.shard_rows(T, rank, world)
    local_mean, _ = oracle.ce_f32(z[lo:hi], t[lo:hi])
    mean = lmdist.combine_mean(local_mean, hi - lo)
    slowest = lmdist.max_over_ranks(float(rank + 1))
    return mean, slowest


def test_token_sharded_mean_over_gloo_ranks():
    out = spawn(_token_sharded)
    T, V = 37, 300
    want, _ = oracle.ce_f32(gen.normal_f32(3, 0, (T, V)), gen.targets(3, 1, (T,), V))
    for rank, (mean, slowest) in out.items():
        assert mean == pytest.approx(want, rel=1e-13)
        assert slowest == 2.0


def _vocab_parallel(rank, world):
    """Each rank: the oracle's partials of its own vocab shard (the rank's
    local logits only), the exchange through dist.gather_partials, and the
    oracle's merge of the gathered block."""
    S, B, V = 5, 3, 1001
    z = gen.normal_bf16_bits(4, 0, (S, B, V), sigma=3.0)
    t = gen.targets(4, 1, (S, B), V)
    v0, w = lmdist.shard_vocab(V, rank, world)
    local = np.ascontiguousarray(z[..., v0:v0 + w])
    m, s, zt = oracle.ce_partials_bf16(local, t, v0)
    part = torch.from_numpy(np.stack([m, s, zt]))
    gathered = lmdist.gather_partials(part).numpy()
    assert gathered.shape == (world, 3, S, B)
    np.testing.assert_array_equal(gathered[rank], part.numpy())   # rank order
    return oracle.ce_merge(gathered[:, 0], gathered[:, 1], gathered[:, 2], t, V)


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_exchange_over_gloo_ranks(world):
    out = spawn(_vocab_parallel, world=world)
    S, B, V = 5, 3, 1001
    want = oracle.ce_sbv_bf16(gen.normal_bf16_bits(4, 0, (S, B, V), sigma=3.0), gen.targets(4, 1, (S, B), V))
    for rank, loss in out.items():
        np.testing.assert_allclose(loss, want, rtol=1e-12, atol=1e-12)


def test_shard_vocab_covers_in_rank_order():
    for V in (1, 7, 128256):
        for world in (1, 2, 3, 8):
            if V < world:
                continue
            shards = [lmdist.shard_vocab(V, r, world) for r in range(world)]
            assert shards[0][0] == 0 and sum(w for _, w in shards) == V
            for (a, wa), (b, _) in zip(shards, shards[1:]):
                assert a + wa == b


def _vp_flce(rank, world):
    """Each rank: the oracle's shard partials of the fused CE from its rows
    of W, the exchange through dist.gather_partials, the oracle's merge."""
    T, H, V = 6, 16, 101
    x = gen.normal_bf16_bits(5, 0, (T, H), sigma=1.0)
    W = gen.normal_bf16_bits(5, 1, (V, H), sigma=0.3)
    t = gen.targets(5, 2, (T,), V)
    v0, w = lmdist.shard_vocab(V, rank, world)
    m, s, zt = oracle.flce_partials_bf16(x, np.ascontiguousarray(W[v0:v0 + w]), t, v0)
    g = lmdist.gather_partials(torch.from_numpy(np.stack([m, s, zt]))).numpy()
    assert g.shape == (world, 3, T)
    return oracle.ce_merge(g[:, 0], g[:, 1], g[:, 2], t, V)


def _vp_fljsd(rank, world):
    """Each rank: its heads' rows, the two exchanges of dist.vocab_parallel_fljsd
    (log-sum-exps [2, T], then term sums [1, T]) with the oracle's shard steps."""
    T, H, V = 7, 16, 89
    xs = gen.normal_bf16_bits(6, 0, (T, H), sigma=1.0)
    Ws = gen.normal_bf16_bits(6, 1, (V, H), sigma=0.3)
    xt = gen.normal_bf16_bits(6, 2, (T, H), sigma=1.0)
    Wt = gen.normal_bf16_bits(6, 3, (V, H), sigma=0.3)
    keep = (np.arange(T) % 3 != 2).astype(np.uint8)
    v0, w = lmdist.shard_vocab(V, rank, world)
    a, b = np.ascontiguousarray(Ws[v0:v0 + w]), np.ascontiguousarray(Wt[v0:v0 + w])
    lse_local = oracle.fljsd_lse_shard_bf16(xs, a, xt, b, 1.5)
    lse = oracle.lse_merge(lmdist.gather_partials(torch.from_numpy(lse_local)).numpy())
    terms = oracle.fljsd_terms_shard_bf16(xs, a, xt, b, lse, 0.3, 1.5)
    allt = lmdist.gather_partials(torch.from_numpy(terms).view(1, T)).view(-1, T).numpy()
    assert allt.shape == (world, T)
    return oracle.jsd_merge(allt, keep)


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_fused_exchanges_over_gloo_ranks(world):
    out = spawn(_vp_flce, world=world)
    T, H, V = 6, 16, 101
    _, want = oracle.flce_bf16(gen.normal_bf16_bits(5, 0, (T, H), sigma=1.0),
                               gen.normal_bf16_bits(5, 1, (V, H), sigma=0.3), gen.targets(5, 2, (T,), V))
    for loss in out.values():
        np.testing.assert_allclose(loss, want, rtol=1e-12, atol=1e-12)
    out = spawn(_vp_fljsd, world=world)
    T, H, V = 7, 16, 89
    want_mean, want_rows = oracle.fljsd_ex_bf16(
        gen.normal_bf16_bits(6, 0, (T, H), sigma=1.0), gen.normal_bf16_bits(6, 1, (V, H), sigma=0.3),
        gen.normal_bf16_bits(6, 2, (T, H), sigma=1.0), gen.normal_bf16_bits(6, 3, (V, H), sigma=0.3), 0.3, 1.5,
        (np.arange(T) % 3 != 2).astype(np.uint8))
    for mean, rows in out.values():
        np.testing.assert_allclose(rows, want_rows, rtol=1e-11, atol=1e-15)
        assert mean == pytest.approx(want_mean, rel=1e-11)


def _vp_flce_bwd(rank, world):
    """Each rank: its shard's forward partials, their all-gather, the oracle's
    shard gradient with the global normalisers from the gathered partials,
    and the all-reduce of the dx shares that dist.vocab_parallel_flce_fwd_bwd
    makes; returns (dx, this rank's dW rows, its vocab range)."""
    T, H, V = 5, 16, 71
    x = gen.normal_bf16_bits(8, 0, (T, H), sigma=1.0)
    W = gen.normal_bf16_bits(8, 1, (V, H), sigma=0.3)
    t = gen.targets(8, 2, (T,), V)
    v0, w = lmdist.shard_vocab(V, rank, world)
    Wl = np.ascontiguousarray(W[v0:v0 + w])
    m, s, zt = oracle.flce_partials_bf16(x, Wl, t, v0)
    g = lmdist.gather_partials(torch.from_numpy(np.stack([m, s, zt]))).numpy()
    lse = oracle.ce_partials_lse(g[:, 0], g[:, 1])
    dx, dW = oracle.flce_grad_shard_bf16(x, Wl, t, v0, V, lse, 0.8)
    dxt = torch.from_numpy(dx)
    dist.all_reduce(dxt, op=dist.ReduceOp.SUM)
    return dxt.numpy(), dW, (v0, w)


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_flce_backward_exchange_over_gloo_ranks(world):
    out = spawn(_vp_flce_bwd, world=world)
    T, H, V = 5, 16, 71
    dx_want, dW_want = oracle.flce_grad_bf16(gen.normal_bf16_bits(8, 0, (T, H), sigma=1.0),
                                             gen.normal_bf16_bits(8, 1, (V, H), sigma=0.3),
                                             gen.targets(8, 2, (T,), V), 0.8)
    for dx, dW, (v0, w) in out.values():
        np.testing.assert_allclose(dx, dx_want, rtol=1e-11, atol=1e-15)
        np.testing.assert_allclose(dW, dW_want[v0:v0 + w], rtol=1e-11, atol=1e-15)


def _vp_fljsd_bwd(rank, world):
    """The student backward's exchanges (log-sum-exps, then JSD terms and KL
    shares in one [2, T] block, then the all-reduce of the dx shares), each
    rank's steps done by the oracle."""
    T, H, V = 5, 16, 67
    xs = gen.normal_bf16_bits(9, 0, (T, H), sigma=1.0)
    Ws = gen.normal_bf16_bits(9, 1, (V, H), sigma=0.3)
    xt = gen.normal_bf16_bits(9, 2, (T, H), sigma=1.0)
    Wt = gen.normal_bf16_bits(9, 3, (V, H), sigma=0.3)
    keep = (np.arange(T) != 3).astype(np.uint8)
    v0, w = lmdist.shard_vocab(V, rank, world)
    a, b = np.ascontiguousarray(Ws[v0:v0 + w]), np.ascontiguousarray(Wt[v0:v0 + w])
    lse = oracle.lse_merge(lmdist.gather_partials(torch.from_numpy(oracle.fljsd_lse_shard_bf16(xs, a, xt, b, 1.2)))
                           .numpy())
    tk = np.stack([oracle.fljsd_terms_shard_bf16(xs, a, xt, b, lse, 0.4, 1.2),
                   oracle.fljsd_kl_shard_bf16(xs, a, xt, b, lse, 0.4, 1.2)])
    allp = lmdist.gather_partials(torch.from_numpy(tk)).numpy()
    kl = allp[:, 1].sum(axis=0)
    dx, dW = oracle.fljsd_grad_shard_bf16(xs, a, xt, b, lse, kl, 0.4, 1.2, keep, 1.1)
    dxt = torch.from_numpy(dx)
    dist.all_reduce(dxt, op=dist.ReduceOp.SUM)
    return dxt.numpy(), dW, (v0, w)


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_fljsd_backward_exchanges_over_gloo_ranks(world):
    out = spawn(_vp_fljsd_bwd, world=world)
    T, H, V = 5, 16, 67
    dx_want, dW_want = oracle.fljsd_grad_bf16(
        gen.normal_bf16_bits(9, 0, (T, H), sigma=1.0), gen.normal_bf16_bits(9, 1, (V, H), sigma=0.3),
        gen.normal_bf16_bits(9, 2, (T, H), sigma=1.0), gen.normal_bf16_bits(9, 3, (V, H), sigma=0.3), 0.4, 1.2,
        (np.arange(T) != 3).astype(np.uint8), 1.1)
    for dx, dW, (v0, w) in out.values():
        np.testing.assert_allclose(dx, dx_want, rtol=1e-10, atol=1e-15)
        np.testing.assert_allclose(dW, dW_want[v0:v0 + w], rtol=1e-10, atol=1e-15)


def _vp_flat(rank, world):
    T, V = 7, 301
    z = gen.normal_f32(10, 0, (T, V))
    t = gen.targets(10, 1, (T,), V)
    v0, w = lmdist.shard_vocab(V, rank, world)
    m, s, zt = oracle.ce_partials_f32(np.ascontiguousarray(z[:, v0:v0 + w]), t, v0)
    g = lmdist.gather_partials(torch.from_numpy(np.stack([m, s, zt]))).numpy()
    return oracle.ce_merge(g[:, 0], g[:, 1], g[:, 2], t, V)


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_flat_exchange_over_gloo_ranks(world):
    out = spawn(_vp_flat, world=world)
    _, want = oracle.ce_f32(gen.normal_f32(10, 0, (7, 301)), gen.targets(10, 1, (7,), 301))
    for loss in out.values():
        np.testing.assert_allclose(loss, want, rtol=1e-12, atol=1e-12)
