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


def _gather(partial: torch.Tensor) -> torch.Tensor:
    """Every rank's FP32 vector, rank r in row r of a [world, N] tensor."""
    world = dist.get_world_size()
    parts = torch.empty((world, partial.numel()), dtype=partial.dtype, device=partial.device)
    if partial.is_cuda:
        dist.all_gather_into_tensor(parts, partial.contiguous())
    else:
        dist.all_gather(list(parts.unbind(0)), partial.contiguous())
    return parts


def _multi() -> bool:
    return dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1


def combine_partials(partial: torch.Tensor) -> torch.Tensor:
    """Sum of every rank's partial dW / dB vector (FP32), added in rank order
    0, 1, ... on every rank (deterministic: the same bits on all ranks and in
    every run)."""
    out = torch.empty_like(partial)
    return combine_into(partial, out)


def combine_into(partial: torch.Tensor, out: torch.Tensor) -> torch.Tensor:
    """The rank-order sum of every rank's FP32 `partial`, converted once into
    `out` (FP32 or the weight's 16-bit type).  On CUDA tensors the sum and
    the conversion are one kernel of the library (norm_sum_ranks) after an
    all-gather; CPU tensors -- the gloo runs that test this host logic on
    machines without a GPU -- add the gathered rows in the same order with
    torch."""
    if partial.is_cuda:
        from . import _binding as B
        parts = _gather(partial) if _multi() else partial.reshape(1, -1)
        if not _multi() and out.data_ptr() == partial.data_ptr():
            return out   # one rank, FP32: the partial is the result
        B.norm_sum_ranks(parts, out)
        return out
    if not _multi():
        if out.data_ptr() != partial.data_ptr():
            out.copy_(partial)
        return out
    parts = _gather(partial)
    total = parts[0].clone()
    for p in parts[1:]:
        total += p
    out.copy_(total)
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
