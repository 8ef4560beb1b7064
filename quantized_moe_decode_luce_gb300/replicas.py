"""Replica bookkeeping for runs on several GPUs of one node.

The decode step does not shard across devices here: every rank runs the whole
path on inputs of its own (a seed per rank), with no collective on the data
path.  The job's time is the maximum of the ranks' device times, and its
throughput counts the units of every rank (weak scaling).
"""
from __future__ import annotations


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's inputs: distinct per rank, the same on every run."""
    return seed * 1000 + rank


def job_throughput(local_ms: float, units_per_rank: int, world: int, device) -> tuple[float, float]:
    """(units per second of the whole job, the slowest rank's ms).

    Every rank calls it with its own timed region; with world > 1 the ranks
    agree on the maximum through one all-reduce of a single number (host
    bookkeeping, not part of the timed work)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    return units_per_rank * world / (ms / 1e3), ms
