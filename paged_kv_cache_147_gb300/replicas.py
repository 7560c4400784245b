"""Data-parallel replicas: one process per GPU, each decoding its own batch.

Decode attention shards by sequence with no exchange between shards, so N GPUs run N
independent replicas and the only cross-process step is the timing reduction: the job's
time is the slowest rank's, and its work is the sum of the ranks' work.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def world() -> tuple[int, int, int]:
    """(rank, local_rank, world_size) from the torchrun environment (1 process if unset)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def init(backend: str | None = None) -> None:
    rank, _, ws = world()
    if ws > 1 and not dist.is_initialized():
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)


def barrier() -> None:
    if dist.is_initialized():
        dist.barrier()


def aggregate(elapsed_s: float, work: float, device="cpu") -> tuple[float, float]:
    """(max elapsed over ranks, summed work over ranks)."""
    if not dist.is_initialized():
        return elapsed_s, work
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([work], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def shutdown() -> None:
    if dist.is_initialized():
        dist.destroy_process_group()
