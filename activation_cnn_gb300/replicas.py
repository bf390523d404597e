"""Multi-GPU execution: independent replicas, one process per GPU.

Images are independent through the whole conv stack, so N GPUs run N copies
of the workload on their own batches (weak scaling) with no collective on the
data path.  The only cross-rank traffic is host-side bookkeeping: a barrier
around the timed region and the max over ranks of the elapsed time.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env():
    """(rank, world_size, local_rank) from the torchrun environment (1 process by default)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard(total: int, world: int, rank: int):
    """Contiguous [start, stop) slice of `total` items for `rank`; sizes differ by <= 1."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError((world, rank))
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def _reduce(value: float, op) -> float:
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(value: float) -> float:
    return _reduce(value, dist.ReduceOp.MAX)


def sum_over_ranks(value: float) -> float:
    return _reduce(value, dist.ReduceOp.SUM)


def barrier() -> None:
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()
