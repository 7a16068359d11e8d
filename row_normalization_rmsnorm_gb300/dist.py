"""Multi-GPU runs: one process per GPU, launched by torchrun, rows sharded
by M.

Rows are independent, so a forward needs no exchange between ranks; the
only exchange a sharded backward has is the sum over ranks of the N-length
FP32 dW / dB partials -- the cross-program column reduction of "perf(norm):
skip dW/dB calculation when parameters are frozen" (Motivation), now across
GPUs -- done here in a fixed rank order so the result does not depend on the
collective's own reduction order.  A frozen parameter has no partial and no
exchange.
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


def combine_into(partial: torch.Tensor, out: torch.Tensor) -> torch.Tensor:
    """combine_partials(partial), written (cast once) into `out`."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        if out.data_ptr() != partial.data_ptr():
            out.copy_(partial)
        return out
    out.copy_(combine_partials(partial))
    return out


def sharded_backward(kind: str, dy, x, w, stats, dx, dw=None, db=None, dh_out=None, offset=0.0, eps=1e-6,
                     workspace=None, partials=None):
    """Backward of one M-sharded problem, from this rank's rows.

    kind: "rms", "ln" or "fadd".  dy, x (h for "fadd"), dx and dh_out hold
    this rank's rows (shard_rows); stats is rstd (or (mean, rstd) for "ln")
    of those rows.  dw / db (None = frozen) receive the gradient of the whole
    problem: this rank's column sums are reduced in FP32 by the library
    (into `partials`, FP32 [N] tensors, allocated when not given), then
    summed over ranks in rank order and cast once to dw / db's dtype.  dx is
    this rank's rows only.  Everything runs on the current stream.  Returns
    (dw, db)."""
    from . import _binding as B
    N = x.shape[1]
    multi = dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1

    def part(i, t):
        if t is None:
            return None
        if not multi and t.dtype == torch.float32:
            return t   # one rank: the library's FP32 sum is the result
        if partials is not None and partials[i] is not None:
            return partials[i]
        return torch.empty(N, dtype=torch.float32, device=x.device)

    pw, pb = part(0, dw), part(1, db)
    if kind == "rms":
        B.norm_rms_bwd(dy, x, w, stats, dx, pw, workspace, offset, eps)
    elif kind == "ln":
        mean, rstd = stats
        B.norm_ln_bwd(dy, x, w, mean, rstd, dx, pw, pb, workspace, offset, eps)
    elif kind == "fadd":
        B.norm_fused_add_rms_bwd(dy, dh_out, x, w, stats, dx, pw, workspace, offset, eps)
    else:
        raise ValueError(f"unknown kind {kind!r}")
    if dw is not None:
        combine_into(pw, dw)
    if db is not None:
        combine_into(pb, db)
    return dw, db
