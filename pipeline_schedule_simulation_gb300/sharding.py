"""Host-side sharding of a batch over ranks (one GPU per process).

Instances are independent, so each rank takes a contiguous range and no data
crosses ranks while they are evaluated.  Only the partition search ends with a
reduction: the (makespan, candidate index) pairs of every rank's best are
gathered and the minimum taken, ties to the lower index.
"""
from __future__ import annotations


def shard_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [lo, hi) of n units for `rank` of `world`; sizes differ by <= 1."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def best_of(pairs):
    """Minimum over (makespan, index) pairs; infeasible entries have index < 0."""
    feasible = [(m, i) for m, i in pairs if i >= 0 and m >= 0]
    if not feasible:
        return (-1, -1)
    return min(feasible)


def reduce_best(makespan: int, index: int, group=None) -> tuple[int, int]:
    """Gather every rank's (makespan, index) with torch.distributed and return the
    global best.  Works on any backend (gloo on CPU, nccl on GPU)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    mine = torch.tensor([makespan, index], dtype=torch.int64)
    if dist.get_backend(group) == "nccl":
        mine = mine.cuda()
    got = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(got, mine, group=group)
    return best_of([(int(t[0]), int(t[1])) for t in got])
