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

Shards are cut at multiples of 8 slices where the axis allows (whole outer
groups of both backward group sizes), the last rank taking any remainder.
Every compute step runs in the library's kernels; this module only splits
ranges and moves the FP32 parts.

The same split also bounds memory on one GPU: ``chunked_tri_attn_bwd`` runs
the outer axis in chunks whose FP32 partials fit a workspace cap (the
partials of one call grow as N_o N^2, the reason the pages bound them by
reusing chunked buffers, "TurboPairFormer", Table 2), and combines the
chunks' FP32 dbias parts in order.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist

from . import triattn as T

SHARD_MULTIPLE = 8


def outer_shard(n_outer: int, rank: int, world: int, multiple: int = SHARD_MULTIPLE) -> Tuple[int, int]:
    """Contiguous slice range [lo, hi) of ``rank``.  With at least ``multiple``
    slices per rank the ranges are whole blocks of ``multiple`` slices (the
    first ranks taking one block more when they do not divide evenly) and the
    last rank also takes the ``n_outer % multiple`` slices left over; with
    fewer, the slices are split as evenly as possible.  Every rank gets at
    least one slice."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    if n_outer < world:
        raise ValueError(f"{n_outer} slices cannot give {world} ranks one slice each")
    unit = multiple if n_outer // multiple >= world else 1
    blocks = n_outer // unit
    base, extra = divmod(blocks, world)
    lo_blk = rank * base + min(rank, extra)
    hi_blk = lo_blk + base + (1 if rank < extra else 0)
    hi = n_outer if rank == world - 1 else hi_blk * unit
    return lo_blk * unit, hi


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


def chunk_slices(n_outer: int, bytes_for, max_workspace_bytes: int, multiple: int = SHARD_MULTIPLE) -> int:
    """The largest chunk of outer slices -- a multiple of ``multiple`` below
    ``n_outer``, or ``n_outer`` itself -- whose backward workspace
    ``bytes_for(chunk)`` fits in ``max_workspace_bytes``; raises if none fits."""
    best = 0
    for c in list(range(multiple, n_outer, multiple)) + [n_outer]:
        need = bytes_for(c)
        if need == 0:
            raise ValueError(f"unsupported shape for a chunk of {c} slices")
        if need <= max_workspace_bytes:
            best = c
        else:
            break  # the workspace grows with the chunk
    if best == 0:
        first = min(multiple, n_outer)
        raise ValueError(f"a chunk of {first} slices needs {bytes_for(first)} workspace bytes, "
                         f"more than {max_workspace_bytes}")
    return best


def chunked_tri_attn_bwd(q, k, v, bias, mask, o, o_resid, lse, do, *, max_workspace_bytes: int, stream=None):
    """Backward with a bounded workspace.  The FP32 dQ and dbias partials of
    one call grow with N_o * N^2; this runs the outer axis in consecutive
    chunks (per example) whose workspace fits ``max_workspace_bytes``, one
    workspace reused by every chunk.  dQ, dK and dV are those of the one-call
    backward, bit for bit (slices are independent); dbias is each chunk's FP32
    sum added in chunk order and rounded once (``tri_attn_dbias_combine``), so
    it is reproducible but its FP32 addition order differs from the one-call
    backward's.  Returns (dq, dk, dv, dbias) in BF16."""
    B, No, H, N, D = q.shape

    def bytes_for(c):
        return T.bwd_workspace_bytes(T.Shape(1, c, N, H, D, T.FLAG_DBIAS_FP32))

    chunk = chunk_slices(No, bytes_for, max_workspace_bytes)
    ws = torch.empty(bytes_for(chunk), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    dbias = torch.empty_like(bias)
    for b in range(B):
        parts = []
        for lo in range(0, No, chunk):
            hi = min(No, lo + chunk)
            sl = (slice(b, b + 1), slice(lo, hi))
            part = torch.empty((1, H, N, N), dtype=torch.float32, device=q.device)
            T.tri_attn_bwd(q[sl], k[sl], v[sl], bias[b:b + 1], None if mask is None else mask[sl], o[sl],
                           None if o_resid is None else o_resid[sl], lse[sl], do[sl], workspace=ws,
                           out=(dq[sl], dk[sl], dv[sl], part), stream=stream, dbias_fp32=True)
            parts.append(part)
        T.tri_attn_dbias_combine(torch.stack(parts), out=dbias[b:b + 1], stream=stream)
    return dq, dk, dv, dbias
