"""Host-side data-parallel helpers: blocks are independent, so ranks share no data-path collective.

Each rank runs its own blocks through the library; only the timing summary crosses ranks (one
all-reduce of a few scalars after the timed region).
"""
from __future__ import annotations

from typing import Tuple

import torch
import torch.distributed as dist


def shard_blocks(total_blocks: int, world: int, rank: int) -> Tuple[int, int]:
    """Contiguous, balanced split of `total_blocks` over `world` ranks: (first block, count) of `rank`."""
    if world < 1 or not 0 <= rank < world or total_blocks < 0:
        raise ValueError("bad shard request")
    lo = total_blocks * rank // world
    hi = total_blocks * (rank + 1) // world
    return lo, hi - lo


def aggregate_throughput(local_blocks: int, local_ms: float, device=None) -> Tuple[float, int, float]:
    """(blocks per second of the whole job, total blocks, max time over ranks in ms).

    The whole job's time is the slowest rank's; blocks add up. Works on any initialised process
    group (gloo on CPU tensors, NCCL on CUDA tensors) and without one (single process).
    """
    t = torch.tensor([float(local_blocks), float(local_ms)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        blocks = t[:1].clone()
        ms = t[1:].clone()
        dist.all_reduce(blocks, op=dist.ReduceOp.SUM)
        dist.all_reduce(ms, op=dist.ReduceOp.MAX)
        total_blocks, max_ms = float(blocks.item()), float(ms.item())
    else:
        total_blocks, max_ms = float(t[0]), float(t[1])
    return total_blocks / (max_ms / 1e3), int(round(total_blocks)), max_ms
