"""Process-group plumbing for multi-GPU benchmark runs (one process per GPU).

The KDA hot path shards with no exchange: every (sequence, head) chain is
independent, so each rank runs its own batch and ranks meet only for the
start/stop barrier and the max-over-ranks of the timed interval.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env_world():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def init(backend: str | None = None):
    rank, world, local = env_world()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group(backend, device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return rank, world, local


def barrier():
    if dist.is_initialized():
        dist.barrier()


def _reduce(x: float, op) -> float:
    if not dist.is_initialized():
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(x: float) -> float:
    return _reduce(x, dist.ReduceOp.MAX)


def sum_over_ranks(x: float) -> float:
    return _reduce(x, dist.ReduceOp.SUM)


def shard(n_units: int, rank: int, world: int):
    """Contiguous [begin, end) share of n_units for this rank (sizes differ by at most 1)."""
    base, extra = divmod(int(n_units), int(world))
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def finalize():
    if dist.is_initialized():
        dist.destroy_process_group()
