"""Process-group plumbing for running the layer step on several GPUs of one
node as independent replicas.

The FP8 linear path has no exchange step inside it: each GPU quantizes and
multiplies its own token shard (the Puro-2B pages train with data parallelism
plus pipeline parallelism and no tensor parallelism, blog section on the RTX
5090 cluster).  A weight-gradient all-reduce would follow the step in
training; it belongs to the optimizer, not to this path.  So ranks only need
a barrier around the timed region and a max-reduction of their times.
"""
from __future__ import annotations

import os
from dataclasses import dataclass

import torch
import torch.distributed as dist


@dataclass
class Ranks:
    rank: int
    world: int
    local_rank: int
    initialized: bool


def init_from_env(backend: str) -> Ranks:
    """Join the process group described by torchrun's environment, if any."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return Ranks(rank, world, local, dist.is_initialized())


def barrier(r: Ranks, device=None) -> None:
    if r.initialized:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(r: Ranks, value: float, device=None) -> float:
    """Largest value across ranks (every rank receives it)."""
    if not r.initialized:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if (device is not None and dist.get_backend() == "nccl") else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(r: Ranks, value: float, device=None) -> float:
    if not r.initialized:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if (device is not None and dist.get_backend() == "nccl") else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shutdown(r: Ranks) -> None:
    if r.initialized and dist.is_initialized():
        dist.destroy_process_group()
