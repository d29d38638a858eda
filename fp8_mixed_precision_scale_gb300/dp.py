"""The data-parallel exchange of the delayed-scaling recipe.

With tokens sharded over ranks, each rank's quantize calls max-accumulate
the amax of its own shard into slot 0 of the amax history.  Before the
history update the ranks must agree on the amax of the whole (unsharded)
tensor, which is the maximum over the ranks' slot-0 values; otherwise the
replicas would derive different scales.  This is one MAX all-reduce of n
floats per step (all histories in one message).  The rowwise recipe needs no
exchange.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def reduce_current_amax(hist: torch.Tensor, group=None) -> None:
    """MAX-all-reduce hist[:, 0] (the current step's amax of every tensor) in place."""
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        return
    cur = hist[:, 0].contiguous()
    dist.all_reduce(cur, op=dist.ReduceOp.MAX, group=group)
    hist[:, 0].copy_(cur)
