"""Host-side logic of running the op as independent replicas, one per GPU.

The op has no parameters and every (pixel, group) unit is independent, so a
batch shards by image with no data-path collective: each rank runs its own
batch (weak scaling).  The only cross-rank traffic is the timing reduction
below (a handful of floats), not data.
"""
from __future__ import annotations

import torch


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of rank's synthetic batch: distinct per rank, rank 0 keeps the base."""
    return base_seed + 7919 * rank


def max_over_ranks(values, dist=None, device=None) -> list[float]:
    """Element-wise maximum of per-rank timings (the slowest rank sets the pace)."""
    vals = [float(v) for v in values]
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def aggregate_gbs(bytes_per_rank_step: int, world: int, step_ms: float) -> float:
    """Whole-job throughput: every rank moved its step's bytes in step_ms."""
    return world * bytes_per_rank_step / (step_ms * 1e-3) / 1e9
