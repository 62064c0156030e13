"""Host-side helpers of the multi-process (one process per GPU) mode.

Token sharding: every row's loss depends on that row alone, so N processes
each run the kernels on their own token slice, and what crosses processes is
scalar bookkeeping only:
  * the global mean of a token-sharded batch, from each rank's (sum, count);
  * timing (max over ranks) and barriers for the benchmark.

Vocab sharding (tensor parallelism, page "Vocab-parallel cross-entropy,
Megatron layout": each rank holds the logits of its own vocab range): each
rank reduces its shard to per-token partials (ce_partials_sbv_bf16), one
all-gather puts every rank's partials on every rank in rank order, and each
rank merges them into the per-token losses (ce_merge_partials).  12 bytes
per token per rank cross the link; the logits never do.

The same split of the output layer's rows for the fused losses: the fused CE
exchanges the same 12 bytes per token (flce_partials_bf16); the fused JSD
exchanges twice, each head's log-sum-exp over the shard (8 bytes per token,
then lse_merge_partials) and then the shard's sum of JSD terms (4 bytes per
token, then jsd_merge_terms), since the divergence needs both heads' global
normalisers.

These run over any torch.distributed backend (NCCL between GPUs, gloo on CPU).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_rows(T: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous token slice [lo, hi) of `rank`; slices are disjoint and
    cover [0, T), sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(T, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def _device_of(group):
    backend = dist.get_backend(group)
    return torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")


def combine_mean(local_mean: float, local_count: int, group=None) -> float:
    """Global mean over all ranks' tokens from each rank's mean over its own
    tokens (fp64 all-reduce of sum and count)."""
    t = torch.tensor([float(local_mean) * local_count, float(local_count)], dtype=torch.float64,
                     device=_device_of(group))
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t[0].item() / t[1].item()) if t[1].item() > 0 else float("nan")


def max_over_ranks(x: float, group=None) -> float:
    t = torch.tensor([float(x)], dtype=torch.float64, device=_device_of(group))
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def shard_vocab(V: int, rank: int, world: int) -> tuple[int, int]:
    """(vocab_start, width) of `rank`'s contiguous vocab shard: the shards
    cover [0, V) in rank order, widths differ by at most one."""
    lo, hi = shard_rows(V, rank, world)
    return lo, hi - lo


def gather_partials(part_local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of every rank's shard partials [3, ...] into [world, 3, ...]
    in rank order: the layout ce_merge_partials reads.  One collective."""
    world = dist.get_world_size(group)
    part_local = part_local.contiguous()
    shape = tuple(part_local.shape)
    # concatenated along the first dimension (the form every backend takes), viewed per rank
    out = torch.empty((world * shape[0],) + shape[1:], dtype=part_local.dtype, device=part_local.device)
    dist.all_gather_into_tensor(out, part_local, group=group)
    return out.view((world,) + shape)


def vocab_parallel_ce(logits_local, target, vocab_start: int, V: int, group=None, partials=None, gathered=None):
    """Per-token Megatron-layout cross-entropy [S, B] of logits whose vocab is
    sharded over the ranks of `group`: this rank holds the columns
    [vocab_start, vocab_start + V_local) of the global vocab V, as bf16
    [S, B, V_local]; target [S, B] holds global indices (the same on every
    rank).  Every rank returns the same losses."""
    from lm_head_online_gb300 import ce_merge_partials, ce_partials_sbv_bf16

    part = ce_partials_sbv_bf16(logits_local, target, vocab_start, partials=partials)
    if gathered is None:
        allp = gather_partials(part, group)
    else:   # caller-owned [world, 3, S, B] buffer
        dist.all_gather_into_tensor(gathered.view((-1,) + tuple(part.shape[1:])), part, group=group)
        allp = gathered
    return ce_merge_partials(allp, target, V)


def vocab_parallel_flce(x, W_local, target, vocab_start: int, V: int, group=None, ws=None):
    """Fused linear + CE with the output layer's rows sharded over the ranks
    of `group`: this rank holds W_local = the global rows [vocab_start,
    vocab_start + V_local) of W, bf16 [V_local, H]; x [T, H] bf16 and target
    [T] int64 (global indices) are the same on every rank.  Returns (mean loss
    [1], per-token losses [T]), the same on every rank."""
    from lm_head_online_gb300 import ce_merge_partials, flce_partials_bf16, rows_mean

    T = target.shape[0]
    part = flce_partials_bf16(x, W_local, target, vocab_start, ws=ws)     # [3, T]
    allp = gather_partials(part, group)                                    # [world, 3, T]
    rows = ce_merge_partials(allp.view(allp.shape[0], 3, T, 1), target.view(T, 1), V).view(T)
    return rows_mean(rows), rows


def vocab_parallel_flce_fwd_bwd(x, W_local, target, vocab_start: int, V: int, grad_scale=1.0, group=None,
                                ws=None):
    """vocab_parallel_flce and the gradients of grad_scale * mean loss: returns
    (mean loss [1], per-token losses [T], dx [T, H] fp32 -- the ranks' shares
    summed by one all-reduce, the same on every rank --, dW_local [V_local, H]
    fp32, this rank's rows of dW).  The backward reuses the forward's gathered
    partials for the global normalisers: no further exchange before dx."""
    from lm_head_online_gb300 import (ce_merge_partials, flce_bwd_workspace_bytes, flce_partials_bf16,
                                      flce_shard_bwd_bf16, rows_mean, workspace)

    T, H = x.shape
    if ws is None:
        ws = workspace(flce_bwd_workspace_bytes(T, H, W_local.shape[0]), x.device)
    part = flce_partials_bf16(x, W_local, target, vocab_start, ws=ws)     # [3, T]
    allp = gather_partials(part, group)                                    # [world, 3, T]
    rows = ce_merge_partials(allp.view(allp.shape[0], 3, T, 1), target.view(T, 1), V).view(T)
    dx, dW = flce_shard_bwd_bf16(x, W_local, target, allp, vocab_start, V, grad_scale, ws=ws)
    dist.all_reduce(dx, op=dist.ReduceOp.SUM, group=group)
    return rows_mean(rows), rows, dx, dW


def vocab_parallel_fljsd(xs, Ws_local, xt, Wt_local, beta=0.5, temperature=1.0, keep=None, group=None, ws=None):
    """Fused linear + generalized JSD with both heads' rows sharded over the
    ranks of `group` (Ws_local, Wt_local: this rank's rows [V_local, H] of the
    student and teacher heads, the same vocab range); xs, xt [T, H] and keep
    are the same on every rank.  Returns (batchmean [1], per-token JSD [T])."""
    from lm_head_online_gb300 import fljsd_lse_partials_bf16, fljsd_terms_bf16, jsd_merge_terms, lse_merge_partials

    T = xs.shape[0]
    lse_local = fljsd_lse_partials_bf16(xs, Ws_local, xt, Wt_local, temperature, ws=ws)       # [2, T]
    lse = lse_merge_partials(gather_partials(lse_local, group))                              # [2, T]
    terms = fljsd_terms_bf16(xs, Ws_local, xt, Wt_local, lse, beta, temperature, ws=ws)       # [T]
    all_terms = gather_partials(terms.view(1, T), group).view(-1, T)                         # [world, T]
    return jsd_merge_terms(all_terms, keep)


def vocab_parallel_fljsd_fwd_bwd(xs, Ws_local, xt, Wt_local, beta=0.5, temperature=1.0, keep=None, grad_scale=1.0,
                                 group=None, ws=None):
    """vocab_parallel_fljsd and the student's gradients of grad_scale * loss:
    returns (batchmean [1], per-token JSD [T], dxs [T, H] fp32 -- the ranks'
    shares summed by one all-reduce --, dWs_local [V_local, H] fp32, this
    rank's rows of the student's dW).  The second exchange carries each
    token's KL(P || M) share beside its JSD terms ([2, T] per rank)."""
    from lm_head_online_gb300 import (fljsd_bwd_workspace_bytes, fljsd_lse_partials_bf16, fljsd_shard_bwd_bf16,
                                      fljsd_terms_bf16, jsd_merge_terms, lse_merge_partials, workspace)

    T, H = xs.shape
    if ws is None:
        ws = workspace(fljsd_bwd_workspace_bytes(T, H, Ws_local.shape[0]), xs.device)
    lse_local = fljsd_lse_partials_bf16(xs, Ws_local, xt, Wt_local, temperature, ws=ws)       # [2, T]
    lse = lse_merge_partials(gather_partials(lse_local, group))                              # [2, T]
    tk = torch.empty((2, T), dtype=torch.float32, device=xs.device)                        # terms, KL shares
    fljsd_terms_bf16(xs, Ws_local, xt, Wt_local, lse, beta, temperature, out=tk[0], ws=ws, kl_local=tk[1])
    allp = gather_partials(tk, group)                                                        # [world, 2, T]
    loss, rows = jsd_merge_terms(allp[:, 0].contiguous(), keep)
    _, kl = jsd_merge_terms(allp[:, 1].contiguous())
    dx, dW = fljsd_shard_bwd_bf16(xs, Ws_local, xt, Wt_local, lse, kl, beta, temperature, keep, grad_scale, ws=ws)
    dist.all_reduce(dx, op=dist.ReduceOp.SUM, group=group)
    return loss, rows, dx, dW


def vocab_parallel_ce_f32(logits_local, target, vocab_start: int, V: int, group=None):
    """Flat fp32 cross-entropy with the vocabulary sharded over the ranks of
    `group`: this rank holds logits_local [T, V_local] = the global columns
    [vocab_start, vocab_start + V_local); target [T] global on every rank.
    Returns (mean loss [1], per-token losses [T]), the same on every rank."""
    from lm_head_online_gb300 import ce_merge_partials, ce_partials_f32, rows_mean

    T = target.shape[0]
    part = ce_partials_f32(logits_local, target, vocab_start)             # [3, T]
    allp = gather_partials(part, group)                                    # [world, 3, T]
    rows = ce_merge_partials(allp.view(allp.shape[0], 3, T, 1), target.view(T, 1), V).view(T)
    return rows_mean(rows), rows


def vocab_parallel_flce_cpo(x, W_local, target, vocab_start: int, V: int, B: int, beta=0.1, alpha=1.0, group=None,
                            ws=None, backward=False, grad_scale=1.0):
    """CPO on the fused linear + CE with W's rows sharded over the ranks of
    `group`: x [B * S, H] bf16 (sequence b < B/2 chosen, b + B/2 its rejected
    answer), target [B * S] global.  The per-token losses come from one
    all-gather of the shards' partials, the CPO combination runs on every rank.
    Returns (loss [1], logps [B]), and with backward=True also (dx [T, H],
    summed over the ranks by one all-reduce, dW_local [V_local, H])."""
    from lm_head_online_gb300 import (ce_merge_partials, cpo_combine_rows, flce_bwd_workspace_bytes,
                                      flce_partials_bf16, flce_shard_bwd_bf16, workspace)

    T, H = x.shape
    if ws is None:
        ws = workspace(flce_bwd_workspace_bytes(T, H, W_local.shape[0]), x.device)
    part = flce_partials_bf16(x, W_local, target, vocab_start, ws=ws)     # [3, T]
    allp = gather_partials(part, group)                                    # [world, 3, T]
    rows = ce_merge_partials(allp.view(allp.shape[0], 3, T, 1), target.view(T, 1), V).view(T)
    row_w = torch.empty_like(rows) if backward else None
    loss, logps = cpo_combine_rows(rows, B, beta, alpha, row_w=row_w)
    if not backward:
        return loss, logps
    dx, dW = flce_shard_bwd_bf16(x, W_local, target, allp, vocab_start, V, grad_scale, ws=ws, row_w=row_w)
    dist.all_reduce(dx, op=dist.ReduceOp.SUM, group=group)
    return loss, logps, dx, dW
