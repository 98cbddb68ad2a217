"""Outer-axis split of triangular attention across GPUs.

The N_o outer slices are independent problems that share one pair bias, so a
group of ranks can each own a contiguous shard of them (the bias replicated on
every rank, as the EvoSP-3D section of "MegaFold: Efficient Training of
Next-Generation 3D Attention Protein Models on Cross-Platform GPUs" does for
its sharded attention stages).  The forward, dQ, dK and dV of a shard need
nothing from other ranks.  dbias is the sum over all slices: every rank runs
the backward with its dbias kept in FP32 (the sum over its own slices), the
parts are gathered in rank order, and ``tri_attn_dbias_combine`` adds them in
ascending rank order and rounds once, so every rank holds the same bits and
the result does not depend on how the gather was scheduled.

Shards are whole multiples of 8 slices (both backward group sizes divide
them).  Every compute step runs in the library's kernels; this module only
splits ranges and moves the FP32 parts.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist

from . import triattn as T

SHARD_MULTIPLE = 8


def outer_shard(n_outer: int, rank: int, world: int, multiple: int = SHARD_MULTIPLE) -> Tuple[int, int]:
    """Contiguous slice range [lo, hi) of ``rank``: whole blocks of ``multiple``
    slices, the first ranks taking one block more when they do not divide
    evenly.  Every rank gets at least one block."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    if n_outer % multiple != 0:
        raise ValueError(f"the outer axis ({n_outer}) must be a multiple of {multiple}")
    blocks = n_outer // multiple
    if blocks < world:
        raise ValueError(f"{n_outer} slices cannot give {world} ranks {multiple} slices each")
    base, extra = divmod(blocks, world)
    lo_blk = rank * base + min(rank, extra)
    hi_blk = lo_blk + base + (1 if rank < extra else 0)
    return lo_blk * multiple, hi_blk * multiple


def gather_rank_ordered(t: torch.Tensor, group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """[R, *t.shape]: every rank's ``t``, stacked in rank order."""
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(t.shape), dtype=t.dtype, device=t.device)
    dist.all_gather(list(out.unbind(0)), t.contiguous(), group=group)
    return out


def sharded_tri_attn_bwd(q, k, v, bias, mask, o, o_resid, lse, do, *,
                         group: Optional[dist.ProcessGroup] = None, workspace=None, stream=None):
    """Backward of this rank's shard of the outer axis (q, k, v, o, o_resid,
    lse, do and mask hold only this rank's slices; bias is the full, replicated
    pair bias).  Returns (dq, dk, dv) of the shard and the full dbias (bf16),
    identical on every rank."""
    dq, dk, dv, part = T.tri_attn_bwd(q, k, v, bias, mask, o, o_resid, lse, do, workspace=workspace,
                                      stream=stream, dbias_fp32=True)
    parts = gather_rank_ordered(part, group)
    dbias = T.tri_attn_dbias_combine(parts, stream=stream)
    return dq, dk, dv, dbias
