"""Replica bookkeeping for runs with one process per GPU.

The decode path shards with no exchange step: (sequence, kv head) units are
independent, including each query head's top-K selection, so a run on N GPUs
is N independent replicas, each running the whole workload on its own GPU
(weak scaling).  The only cross-rank operations are the barriers around the
timed region and the maximum over ranks of its duration, both here; the data
path has no collective.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def rank_info(env=None) -> tuple[int, int, int]:
    """(world size, rank, local rank) from the launcher's environment."""
    env = os.environ if env is None else env
    return (int(env.get("WORLD_SIZE", "1")), int(env.get("RANK", "0")),
            int(env.get("LOCAL_RANK", "0")))


def init(world_size: int, backend: str = "nccl", device: torch.device | None = None):
    """Join the process group when there is more than one rank."""
    if world_size > 1 and not dist.is_initialized():
        if device is not None and backend == "nccl":
            dist.init_process_group(backend, device_id=device)
        else:
            dist.init_process_group(backend)


def barrier(world_size: int):
    if world_size > 1:
        dist.barrier()


def max_over_ranks(x: float, world_size: int, device: str | torch.device = "cpu") -> float:
    """The largest x over all ranks (the slowest replica's time)."""
    if world_size <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds: float, world_size: int) -> float:
    """Units processed by all replicas per second of the slowest one."""
    return world_size * units_per_rank / seconds


def finish(world_size: int):
    if world_size > 1 and dist.is_initialized():
        dist.barrier()
        dist.destroy_process_group()
