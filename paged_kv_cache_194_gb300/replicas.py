"""Multi-GPU replicas of the decode batch.

Sequences are independent, so N GPUs serve N batches with no data-path
collective: rank r draws its own batch (the workload's seed offset by r) and
the only cross-rank traffic is the timing reduction (max over ranks) and the
byte total (sum over ranks).  Works with any torch.distributed backend (nccl
on GPUs, gloo for the host-only tests).
"""
from __future__ import annotations

import dataclasses

import torch
import torch.distributed as dist

from . import workloads as wl

RANK_SEED_STRIDE = 1000


def rank_workload(w: wl.Workload, rank: int) -> wl.Workload:
    """The batch rank `rank` serves (rank 0 serves the workload itself)."""
    return w if rank == 0 else dataclasses.replace(w, seed=w.seed + RANK_SEED_STRIDE * rank)


def _reduce(value: float, op, device) -> float:
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(value: float, device="cpu") -> float:
    return _reduce(value, dist.ReduceOp.MAX, device)


def sum_over_ranks(value: float, device="cpu") -> float:
    return _reduce(value, dist.ReduceOp.SUM, device)
