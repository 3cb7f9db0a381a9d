"""Host logic of the multi-GPU mode: independent replicas.

The M solves of a batch are independent and the path has no exchange step,
so N GPUs run N replicas of the single-GPU path, one process each, on
disjoint slices of the problem stream (weak scaling: every rank solves its
own batch of M).  The only collective is the timing reduction: the job's
time is the slowest rank's, and its throughput is all ranks' solves over
that time.  Everything here is plain host code over torch.distributed, so
it runs on gloo (CPU) as well as NCCL.
"""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class Replica:
    world: int
    rank: int
    local: int

    def first_solve(self, batch: int) -> int:
        """Index of this rank's first solve in the global problem stream."""
        return self.rank * batch

    def solves(self, batch: int) -> range:
        return range(self.first_solve(batch), self.first_solve(batch) + batch)


def from_env() -> Replica:
    """RANK / WORLD_SIZE / LOCAL_RANK as torchrun sets them (1 rank otherwise)."""
    return Replica(world=int(os.environ.get("WORLD_SIZE", "1")),
                   rank=int(os.environ.get("RANK", "0")),
                   local=int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of a list of floats over all ranks (the values
    unchanged with a single rank)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(solves_per_rank: int, world: int, slowest_ms: float) -> float:
    """Whole-job solves per second: every rank's solves over the slowest
    rank's time."""
    return solves_per_rank * world / (slowest_ms / 1000.0)
