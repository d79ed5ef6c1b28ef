"""Data-parallel exchange of the LoRA gradients.

The frozen NF4 weight is identical on every rank (quantisation is
deterministic), so data parallelism over tokens needs one collective per
step: the sum of dA [r, K] and dB [N, r] over ranks.  Y and dX stay local.
This is the only exchange of the path; it runs through torch.distributed
(NCCL on GPUs, gloo on CPU) on the caller's process group.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


def allreduce_lora_grads(da: torch.Tensor, db: torch.Tensor, group=None, average: bool = False) -> None:
    """In-place sum (or mean) of dA and dB over the ranks of `group`.

    Both tensors are packed into one flat buffer so the step issues a single
    collective; the result is written back in place.
    """
    world = dist.get_world_size(group)
    if world == 1:
        return
    flat = torch.cat([da.reshape(-1), db.reshape(-1)])
    dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
    if average:
        flat.div_(world)
    da.copy_(flat[: da.numel()].view_as(da))
    db.copy_(flat[da.numel():].view_as(db))


def shard_tokens(m: int, rank: int, world: int) -> slice:
    """Contiguous token range of `rank` when m tokens are split over `world` ranks."""
    base, extra = divmod(m, world)
    start = rank * base + min(rank, extra)
    return slice(start, start + base + (1 if rank < extra else 0))
