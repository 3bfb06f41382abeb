"""Whole-matrix ownership across ranks.

Newton-Schulz acts on whole matrices, so a data-parallel job gives each rank
complete matrices and runs their steps with no communication ("Training a
1T-Params MoE on EU public infrastructure", tanhow.com, the FlexShard
paragraph: each rank owns whole experts).  ``owner_partition`` decides who
owns what, balancing the step's work; nothing else is exchanged.
"""
from __future__ import annotations

from .workloads import symmetric_flops


def owner_partition(shapes, world: int, iters: int = 5):
    """Rank owning each matrix: longest-processing-time-first on the step's
    symmetric FLOPs (ties broken by matrix index, then by the lowest rank),
    so the result is deterministic and identical on every rank."""
    if world < 1:
        raise ValueError("world must be >= 1")
    cost = [symmetric_flops(r, c, iters) if r and c else 0.0 for r, c in shapes]
    order = sorted(range(len(shapes)), key=lambda i: (-cost[i], i))
    load = [0.0] * world
    owner = [0] * len(shapes)
    for i in order:
        rank = min(range(world), key=lambda k: (load[k], k))
        owner[i] = rank
        load[rank] += cost[i]
    return owner


def owned_indices(shapes, rank: int, world: int, iters: int = 5):
    owner = owner_partition(shapes, world, iters)
    return [i for i, o in enumerate(owner) if o == rank]


def rank_loads(shapes, world: int, iters: int = 5):
    owner = owner_partition(shapes, world, iters)
    load = [0.0] * world
    for (r, c), o in zip(shapes, owner):
        load[o] += symmetric_flops(r, c, iters) if r and c else 0.0
    return load
