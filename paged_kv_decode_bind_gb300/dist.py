"""Host logic for running decode replicas on several GPUs.

Requests are independent, so the path shards by request with no exchange
step: each rank owns a disjoint set of requests (its own pool, table and
workspace) and runs the same kernels.  The only collectives are host-side
bookkeeping for measurement: a barrier, the maximum of the ranks' times and
the sum of their work.
"""
from __future__ import annotations


def shard_range(n_items: int, rank: int, world: int):
    """Contiguous [lo, hi) share of n_items for rank (sizes differ by <= 1)."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(n_items, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def rank_seed(base_seed: int, rank: int) -> int:
    """Distinct input seed per replica."""
    return base_seed + 1000 * rank


def reduce_time_and_work(seconds: float, work: float, device=None):
    """(max over ranks of seconds, sum over ranks of work); identity when
    torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(seconds), float(work)
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    w = torch.tensor([work], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(w, op=dist.ReduceOp.SUM)
    return float(t.item()), float(w.item())
