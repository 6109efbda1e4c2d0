"""Data-parallel replicas of the Engram lookup (host-side helpers).

Every token of the lookup is independent (its row ids depend on its own
4-id window, its streams on its own rows), so N GPUs scale it with no
collective on the data path: each GPU holds a replica of the tables and
processes its own batch (weak scaling), or its contiguous share of one global
batch (strong scaling).  The only cross-rank traffic is control: a barrier
around the timed region and the maximum step time.  These helpers work with any
torch.distributed backend (NCCL on GPUs, gloo in the CPU tests).
"""
from __future__ import annotations


def shard_range(n_items: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced [start, stop) share of n_items for `rank` of `world`.
    The first n_items % world ranks take one extra item."""
    if world < 1 or not 0 <= rank < world or n_items < 0:
        raise ValueError(f"bad shard: n_items={n_items} rank={rank} world={world}")
    base, extra = divmod(n_items, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank scalar (the step time) over the default group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_throughput(tokens_all_ranks: float, seconds_max: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    if seconds_max <= 0:
        raise ValueError("non-positive time")
    return tokens_all_ranks / seconds_max
