"""Multi-GPU bookkeeping for independent layer replicas.

The MoE FFN layer has no exchange step between tokens, so N GPUs run N
independent replicas, each on its own batch of tokens (weak scaling).  Only
the timing is combined: the job's step time is the slowest rank's, and the
job throughput counts every rank's tokens.  These helpers take a
torch.distributed process group (NCCL on GPUs, gloo in the CPU tests).
"""
from __future__ import annotations


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a scalar over all ranks of the default process group."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(local_total_ms: float, tokens_per_rank_step: int, steps: int, world: int,
                   device=None):
    """(tokens/s of the whole job, ms per step) from each rank's own total.

    Every rank passes the device time it measured over `steps` steps; the job
    time is the maximum over ranks (the slowest replica bounds the job).
    """
    total_ms = max_over_ranks(local_total_ms, device)
    tokens = tokens_per_rank_step * steps * world
    return tokens / (total_ms / 1e3), total_ms / steps


def shard_range(n: int, rank: int, world: int):
    """Contiguous [start, stop) share of n items for `rank` (sizes differ by <= 1)."""
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)
