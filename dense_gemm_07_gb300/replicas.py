"""Replica bookkeeping for multi-GPU benchmark runs.

GEMM shards over tiles of C with no exchange between devices, so a run on N
GPUs is N independent replicas of the same step: there is no collective on
the data path.  The only cross-rank communication is the timing contract:
every rank measures its own step time, the job's time is the maximum over
ranks, and whole-job throughput is the work of all ranks divided by it.
"""
from __future__ import annotations


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (identity when
    torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist

    vals = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(world_size: int, work_per_rank_step: float, step_seconds: float) -> float:
    """Work of all ranks per second, given the max-over-ranks step time."""
    if step_seconds <= 0:
        raise ValueError("step time must be positive")
    return world_size * work_per_rank_step / step_seconds
