"""Host logic for running the attention forward on several GPUs of one node.

The work units (sequence b, head h, query tile) are independent: no unit reads
another's output and the per-head outputs are concatenated by layout alone
("Attention Is All You Need", Section 3.2.2; cookipedia article, section
"Transformer の構造").  So ranks share no data and need no collective on the
data path.  Benchmarks use weak scaling: each rank owns a fixed batch of
sequences (its own replica of the workload, drawn with a rank-specific seed),
and the only communication is timing (a barrier and a max over ranks).
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def env_rank_world():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend: str) -> tuple[int, int]:
    """Join the process group when launched with more than one rank."""
    rank, world, _ = env_rank_world()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def shard(total: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [start, stop) share of ``total`` units for ``rank``; shares
    differ by at most one unit and cover 0 .. total-1 exactly once."""
    base, extra = divmod(total, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's replica (rank 0 keeps the workload's own seed)."""
    return seed + 7919 * rank


def barrier(device=None):
    if dist.is_available() and dist.is_initialized():
        if dist.get_backend() == "nccl" and device is not None:
            dist.barrier(device_ids=[device.index if hasattr(device, "index") else int(device)])
        else:
            dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of ``x`` over all ranks (x itself with one rank)."""
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


def finish():
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
