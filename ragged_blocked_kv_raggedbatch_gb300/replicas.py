"""Ranks of a multi-GPU run: one batch per rank, no collective on the data path.

Sequences are independent (each owns its tokens, blocks and work), so N GPUs
run N batches side by side -- the replica parallelism of "DeepSpeed-MII: A
Source Tour" (pyshine.com/deepspeed-mii), section "Under the Load Balancer":
replicas are symmetric and requests independent.  The only communication is
measurement: a barrier before and after the timed region and the maximum of
the ranks' times.
"""
from __future__ import annotations

import os
from typing import Optional, Tuple


def env() -> Tuple[int, int, int]:
    """(world_size, rank, local_rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(seed: int, rank: int) -> int:
    """Seed of the values of rank `rank`'s batch (same structure, own values)."""
    return int(seed) + 7919 * int(rank)


class Group:
    """torch.distributed process group for barrier + max-over-ranks, or a
    no-op stand-in for a single rank."""

    def __init__(self, backend: str = "nccl"):
        self.world, self.rank, self.local = env()
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            if not dist.is_initialized():
                dist.init_process_group(backend)
            self.dist = dist

    def barrier(self) -> None:
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float, device: Optional[str] = None) -> float:
        if self.dist is None:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self) -> None:
        if self.dist is not None:
            self.dist.barrier()
            self.dist.destroy_process_group()
            self.dist = None
