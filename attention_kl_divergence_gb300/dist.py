"""Multi-GPU plumbing for the attention KL divergence.

Every (batch, head) pair is an independent problem for the forward and both
backward settings, so the work shards by heads with no collective on the data
path: each rank owns a contiguous range of flat heads b*H + h and runs the
kernels on it; only timing (a barrier and a max over ranks) crosses ranks.
One process per GPU; the rank/world come from the torchrun environment.
"""
from __future__ import annotations

import os

import torch


def env():
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(world: int, backend: str) -> None:
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def head_range(num_heads: int, rank: int, world: int):
    """[start, stop) of the flat heads rank owns; shards differ by at most one head."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(num_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_heads(t: torch.Tensor, rank: int, world: int) -> torch.Tensor:
    """The rank's heads of a [B, H, N, ...] tensor as a [1, n, N, ...] view
    (B and H flattened; the view keeps the d-contiguous layout)."""
    B, H = t.shape[:2]
    start, stop = head_range(B * H, rank, world)
    return t.reshape(B * H, *t.shape[2:])[start:stop].unsqueeze(0)


def barrier(world: int) -> None:
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())
