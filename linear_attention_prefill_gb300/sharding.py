"""Host-side logic for running the forward on several GPUs, one process each.

Every (sequence, v head) chain is independent across all operators
("Empowering Hybrid Attention Models on NPUs", §4, Insight 1: heads share no
state), so several GPUs split the work without any collective on the data
path: each rank takes whole sequences and writes its own outputs.  The only
communication is the timing reduction of a benchmark (max over ranks).
"""
from __future__ import annotations

import heapq
from typing import List, Sequence


def partition_sequences(seqlens: Sequence[int], world: int) -> List[List[int]]:
    """Split sequence indices over ``world`` ranks, balancing tokens (longest first).

    Every index appears exactly once; ranks may get none when there are fewer
    sequences than ranks.  Each rank's list is in ascending order.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    heap = [(0, r) for r in range(world)]
    parts: List[List[int]] = [[] for _ in range(world)]
    for i in sorted(range(len(seqlens)), key=lambda i: (-int(seqlens[i]), i)):
        load, r = heapq.heappop(heap)
        parts[r].append(i)
        heapq.heappush(heap, (load + int(seqlens[i]), r))
    return [sorted(p) for p in parts]


def rank_seed(seed: int, rank: int) -> int:
    """Seed of rank ``rank``'s own batch when every rank runs the same workload."""
    return seed + 1_000_003 * rank


def reduce_timing(ms: float, units: float, group=None):
    """(max over ranks of ms, sum over ranks of units) through torch.distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return ms, units
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else None
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())
