"""Host-side logic of multi-GPU runs: one process per GPU, launched by
torchrun, rows sharded by M.

Rows are independent, so a forward needs no exchange between ranks; the
only exchange a sharded backward has is the sum over ranks of the N-length
FP32 dW / dB partials, done here in a fixed rank order so the result does
not depend on the collective's own reduction order.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def rank_env():
    """(world_size, rank, local_rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_rows(M: int, rank: int, world: int):
    """Contiguous row range [start, stop) of `rank`: sizes differ by at most
    one row and the ranges partition [0, M)."""
    if world < 1 or not 0 <= rank < world or M < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(M, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank scalar (e.g. a step time) over all ranks."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def combine_partials(partial: torch.Tensor) -> torch.Tensor:
    """Sum of every rank's partial dW / dB vector, added in rank order 0, 1,
    ... on every rank (deterministic: the same bits on all ranks and in
    every run)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return partial.clone()
    parts = [torch.empty_like(partial) for _ in range(dist.get_world_size())]
    dist.all_gather(parts, partial.contiguous())
    total = parts[0].clone()
    for p in parts[1:]:
        total += p
    return total
