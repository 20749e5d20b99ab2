"""Data-parallel replicas: one process per GPU, each with its own copy of the
model, serving its own share of the requests.

Requests are independent and the invariant kernels read neither the batch nor
the SM count, so a request's tokens do not depend on which replica serves it
or with whom: sharding needs no collective on the data path.  The only
cross-rank traffic is host-side bookkeeping — gathering results and taking the
slowest rank's time for throughput.  Works with any torch.distributed backend
(gloo on CPU, NCCL on GPUs).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard(n_items: int, world: int, rank: int) -> list:
    """Round-robin share of items 0..n_items-1 for `rank` of `world`."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad rank {rank} of world {world}")
    return list(range(rank, n_items, world))


def gather(local: dict) -> dict:
    """Union of every rank's {key: value} results, on every rank."""
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return dict(local)
    parts = [None] * dist.get_world_size()
    dist.all_gather_object(parts, local)
    out = {}
    for p in parts:
        overlap = set(out) & set(p)
        if overlap:
            raise ValueError(f"keys served by two replicas: {sorted(overlap)[:5]}")
        out.update(p)
    return out


def max_over_ranks(value: float, device=None) -> float:
    """The slowest rank's value (whole-job time is set by the last replica)."""
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
