"""Host-side helpers of the multi-process (one process per GPU) mode.

The losses shard by tokens with no data exchange: every row's loss depends on
that row alone, so N processes each run the kernels on their own token slice.
What crosses processes is scalar bookkeeping only:
  * the global mean of a token-sharded batch, from each rank's (sum, count);
  * timing (max over ranks) and barriers for the benchmark.
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
