"""Sharding of the head-wise recurrence over GPUs (one process per GPU).

Heads are independent (block-diagonal recurrent matrix, FlashRNN blog page,
head-wise paragraph) and so are batch rows, so the forward shards over either
with no exchange at all: every rank runs its own slice through rnn_fwd.  The
time axis never shards (each step needs the previous one).

Training sharded over the batch needs one exchange after the reverse pass:
dR and db are sums over batch rows, so each rank's partial sums are added with
an all-reduce.  Sharding over heads needs none (each rank owns its heads'
dR/db outright).  The helpers below work with any torch.distributed backend
(NCCL on GPUs; gloo on CPU in the tests).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced [start, stop) slice of n units (heads or batch rows)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def allreduce_weight_grads(dR: torch.Tensor, db: torch.Tensor, group=None) -> None:
    """Sum the batch-sharded partial weight gradients over all ranks, in place."""
    if dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(dR, op=dist.ReduceOp.SUM, group=group)
        dist.all_reduce(db, op=dist.ReduceOp.SUM, group=group)


def max_over_ranks(value: float, device=None, group=None) -> float:
    """Largest of a per-rank scalar (step time): the job finishes with its slowest rank."""
    if not dist.is_initialized() or dist.get_world_size(group) == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
