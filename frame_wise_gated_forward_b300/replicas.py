"""Multi-GPU replicas for benchmarking (one process per GPU).

The frame-wise GDN forward shards with no data exchange: batch rows and heads
are independent problems, so N GPUs run N independent sequences (weak
scaling) and the only collectives are the timing barrier and a max-reduce of
the elapsed time.  Nothing on the data path communicates.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env_world():
    """(rank, local_rank, world_size) from the torchrun environment (1 process if unset)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init(backend: str):
    rank, local_rank, world = env_world()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, local_rank, world


def barrier(device=None):
    if dist.is_available() and dist.is_initialized():
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index] if device is not None else None)
        else:
            dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (x itself with one process)."""
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def throughput(units_per_rank: float, steps: int, seconds_max: float, world: int) -> float:
    """Whole-job rate: units all ranks processed divided by the slowest rank's time."""
    return units_per_rank * steps * world / seconds_max


def shutdown():
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
