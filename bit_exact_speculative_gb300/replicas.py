"""Data-parallel replicas: one process per GPU, each with the whole model and its own sequences.

The verify path shards over independent sequences with no exchange between
them, so N GPUs run N replicas and need no collective on the data path; the
only communication is the timing reduction of a measurement: the job's time
is the slowest rank's, and its work the sum of every rank's.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

# Stride between the sequence seeds of consecutive ranks (a prime, so that rank seeds of
# different base seeds rarely collide).
RANK_SEED_STRIDE = 1_000_003


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of the sequences (caches, states, drafts) of ``rank``: every rank verifies its own."""
    return int(base_seed) + RANK_SEED_STRIDE * int(rank)


def job_throughput(local_seconds: float, local_units: float, device=None):
    """(units of all ranks / slowest rank's seconds, slowest seconds, total units).  Collective over
    the default process group when it is initialised, else this process alone."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_units / local_seconds, float(local_seconds), float(local_units)
    dev = device if device is not None else torch.device("cpu")
    t = torch.tensor([float(local_seconds)], dtype=torch.float64, device=dev)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(u.item()) / float(t.item()), float(t.item()), float(u.item())
