"""Row sharding of one batch across ranks, one process per GPU.

The pages train on 8- and 16-GPU clusters (AdaptiveLoad technical summary, sections 2.A and
4). Rows are independent, so a batch splits into contiguous, segment-aligned row shards,
one per rank: each rank runs the fused forward and backward on its own segments (a packed
call with its slice of the segment table and the batch's modulation tables), which needs
no exchange for y and dx. Its backward gives dshift/dscale over its own tokens only (rows of
the modulation tables its segments do not use come out 0); the batch's gradients are the
sum over ranks. That sum is the one exchange: every rank's [2, nmod, D] fp32 gradients are
gathered and added in rank order 0, 1, ..., world - 1 by ``adaln_sum_ranks``, so every rank
gets the same bits whatever transport moved them (no ring all-reduce, whose summation order
depends on the algorithm and the topology).

torch.distributed only moves bytes here; the arithmetic runs in libadaln's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np


@dataclass
class Shard:
    """Segments [s0, s1) of the batch, i.e. rows [row0, row1)."""
    rank: int
    s0: int
    s1: int
    row0: int
    row1: int
    cu_seqlens: np.ndarray   # int32 [s1 - s0 + 1], starting at 0
    mod_idx: np.ndarray      # int32 [s1 - s0], the batch's modulation rows

    @property
    def rows(self) -> int:
        return self.row1 - self.row0

    @property
    def nseg(self) -> int:
        return self.s1 - self.s0


def plan_shards(cu_seqlens: Sequence[int], world: int) -> List[Tuple[int, int]]:
    """Contiguous segment ranges, one per rank, of about total/world tokens each: rank r's
    range ends at the first segment boundary at or past (r + 1) * total / world tokens.
    Segments are never split, so a rank may get none when segments are few and long."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if world < 1:
        raise ValueError("world must be >= 1")
    nseg = len(cu) - 1
    total = int(cu[-1]) if nseg >= 0 else 0
    bounds = [0]
    for r in range(1, world):
        target = (total * r + world - 1) // world  # ceil(total * r / world)
        bounds.append(max(bounds[-1], int(np.searchsorted(cu, target, side="left"))))
    bounds.append(nseg)
    for i in range(1, len(bounds)):
        bounds[i] = min(max(bounds[i], bounds[i - 1]), nseg)
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def make_shard(cu_seqlens: Sequence[int], mod_idx: Sequence[int], world: int, rank: int) -> Shard:
    """Rank `rank`'s shard: its segment range, row range and local segment table."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    mod = np.asarray(mod_idx, dtype=np.int64)
    s0, s1 = plan_shards(cu, world)[rank]
    row0, row1 = int(cu[s0]), int(cu[s1])
    local_cu = (cu[s0:s1 + 1] - row0).astype(np.int32)
    return Shard(rank, s0, s1, row0, row1, local_cu, mod[s0:s1].astype(np.int32))


def sum_over_ranks(local, group=None, reduce: Optional[Callable] = None):
    """The batch's gradients from every rank's own: `local` is this rank's fp32 tensor
    ([2, nmod, D]: dshift, dscale). Gathers all ranks' tensors and adds them in rank order.
    `reduce(stacked, out, world, n)` performs the ordered sum; the default is libadaln's
    adaln_sum_ranks on the tensors' CUDA device (there is no CPU path in the library)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    local = local.contiguous()
    parts = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(parts, local, group=group)
    stacked = torch.stack(parts)
    out = torch.empty_like(local)
    if reduce is None:
        if not local.is_cuda:
            raise RuntimeError("sum_over_ranks: the library reduces device tensors only")
        from . import adaln_sum_ranks
        adaln_sum_ranks(stacked, out, world, local.numel())
    else:
        reduce(stacked, out, world, local.numel())
    return out
