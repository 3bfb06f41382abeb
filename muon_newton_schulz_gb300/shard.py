"""Whole-matrix ownership across ranks (FlexShard).

Newton-Schulz acts on whole matrices.  "Training a 1T-Params MoE on EU public
infrastructure" (tanhow.com, the FlexShard paragraph) keeps every expert
matrix whole on one rank, which runs its step with no communication, while
the dense matrices stay sharded and are gathered to a rank for their step,
the expert work overlapping that transfer.  "AMD GPU深度学习优化与ZAYA1大模型实践"
(jsqmd.com/news/1098463, section 4.2) moves the shards with point-to-point
sends to the rank that needs them instead of an all-gather to every rank,
which is what cuts the optimizer's peak memory.

``owner_partition`` decides who owns what, balancing the step's work.
``FlexShardPlan`` adds the row shards of the dense matrices, and
``FlexShardStep`` runs one step on a rank: it posts the sends of its dense
shards to their owners and the receives of the shards of the dense matrices
it owns, steps its own experts while those are in flight, steps the gathered
dense matrices, and sends every updated W and M shard back to its holder.
The step itself is a callable (the library's ``MuonStep.step`` on a GPU);
torch.distributed moves the tensors (NCCL on GPUs, gloo on CPUs).
"""
from __future__ import annotations

from dataclasses import dataclass

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


def row_shards(rows: int, world: int):
    """[begin, end) rows held by each rank: contiguous blocks, the first
    rows % world ranks one row longer."""
    base, extra = divmod(rows, world)
    out, b = [], 0
    for k in range(world):
        e = b + base + (1 if k < extra else 0)
        out.append((b, e))
        b = e
    return out


@dataclass(frozen=True)
class FlexShardPlan:
    """Ownership of a batch: ``owner[i]`` runs matrix i's step; a dense matrix
    (``dense[i]``) is held as row shards ``shards[i][k]`` by every rank k."""

    shapes: tuple
    dense: tuple
    world: int
    owner: tuple
    shards: tuple

    @staticmethod
    def build(shapes, dense, world: int, iters: int = 5) -> "FlexShardPlan":
        shapes = tuple((int(r), int(c)) for r, c in shapes)
        dense = tuple(bool(x) for x in dense)
        if len(dense) != len(shapes):
            raise ValueError("one dense flag per matrix")
        owner = tuple(owner_partition(shapes, world, iters))
        shards = tuple(tuple(row_shards(r, world)) if d else None for (r, _), d in zip(shapes, dense))
        return FlexShardPlan(shapes, dense, world, owner, shards)

    def local_shape(self, i: int, rank: int):
        """Shape of what `rank` holds of matrix i: all of an expert it owns,
        its row shard of a dense matrix, nothing (None) otherwise."""
        r, c = self.shapes[i]
        if self.dense[i]:
            b, e = self.shards[i][rank]
            return (e - b, c)
        return (r, c) if self.owner[i] == rank else None

    def experts_of(self, rank: int):
        return [i for i in range(len(self.shapes)) if not self.dense[i] and self.owner[i] == rank]

    def dense_owned_by(self, rank: int):
        return [i for i in range(len(self.shapes)) if self.dense[i] and self.owner[i] == rank]

    def bytes_moved(self, w_bytes: int = 2):
        """Bytes one step sends in total: each dense shard held away from its
        owner travels there as G, M and W (4 + 4 + w_bytes per element) and its
        W and M come back (w_bytes + 4)."""
        total = 0
        for i, (r, c) in enumerate(self.shapes):
            if not self.dense[i]:
                continue
            for k, (b, e) in enumerate(self.shards[i]):
                if k != self.owner[i]:
                    total += (e - b) * c * (4 + 4 + w_bytes + w_bytes + 4)
        return total


class FlexShardStep:
    """One rank's part of a FlexShard step.

    ``step_fn(Ws, Gs, Ms, lrs)`` updates whole matrices in place (W and M);
    ``alloc(shape, dtype)`` makes the owner's gather buffers (on the rank's
    device).  ``local`` maps matrix index -> (W, G, M) of what this rank holds
    (see ``FlexShardPlan.local_shape``)."""

    def __init__(self, plan: FlexShardPlan, rank: int, step_fn, alloc, group=None):
        self.plan = plan
        self.rank = rank
        self.step_fn = step_fn
        self.alloc = alloc
        self.group = group
        self._full = {}

    def _full_buffers(self, i, like):
        if i not in self._full:
            r, c = self.plan.shapes[i]
            W, G, M = like
            self._full[i] = (self.alloc((r, c), W.dtype), self.alloc((r, c), G.dtype), self.alloc((r, c), M.dtype))
        return self._full[i]

    def step(self, local: dict, lrs) -> None:
        import torch.distributed as dist

        plan, me = self.plan, self.rank
        # 1. shards of dense matrices move to their owners (G, M, W in that
        #    order, matrices in index order: both sides issue the same order)
        ops = []
        gathered = {}
        for i in range(len(plan.shapes)):
            if not plan.dense[i]:
                continue
            o = plan.owner[i]
            if o != me:
                W, G, M = local[i]
                for t in (G, M, W):
                    ops.append(dist.P2POp(dist.isend, t.contiguous(), o, self.group))
            else:
                full = self._full_buffers(i, local[i])
                gathered[i] = full
                for k, (b, e) in enumerate(plan.shards[i]):
                    if e == b:
                        continue
                    Wf, Gf, Mf = full
                    if k == me:
                        W, G, M = local[i]
                        Wf[b:e].copy_(W)
                        Gf[b:e].copy_(G)
                        Mf[b:e].copy_(M)
                    else:
                        for t in (Gf, Mf, Wf):
                            ops.append(dist.P2POp(dist.irecv, t[b:e], k, self.group))
        ops = [op for op in ops if op.tensor.numel() > 0]
        reqs = dist.batch_isend_irecv(ops) if ops else []
        # 2. this rank's experts need nothing from anyone: step them while the
        #    dense shards are in flight
        ex = plan.experts_of(me)
        if ex:
            self.step_fn([local[i][0] for i in ex], [local[i][1] for i in ex], [local[i][2] for i in ex],
                         [lrs[i] for i in ex])
        for r in reqs:
            r.wait()
        # 3. the dense matrices this rank owns, whole
        dn = sorted(gathered)
        if dn:
            self.step_fn([gathered[i][0] for i in dn], [gathered[i][1] for i in dn], [gathered[i][2] for i in dn],
                         [lrs[i] for i in dn])
        # 4. updated W and M shards go back to their holders
        ops = []
        for i in range(len(plan.shapes)):
            if not plan.dense[i]:
                continue
            o = plan.owner[i]
            if o != me:
                W, G, M = local[i]
                for t in (W, M):
                    ops.append(dist.P2POp(dist.irecv, t, o, self.group))
            else:
                Wf, Gf, Mf = gathered[i]
                for k, (b, e) in enumerate(plan.shards[i]):
                    if e == b:
                        continue
                    if k == me:
                        W, G, M = local[i]
                        W.copy_(Wf[b:e])
                        M.copy_(Mf[b:e])
                    else:
                        for t in (Wf, Mf):
                            ops.append(dist.P2POp(dist.isend, t[b:e].contiguous(), k, self.group))
        ops = [op for op in ops if op.tensor.numel() > 0]
        for r in (dist.batch_isend_irecv(ops) if ops else []):
            r.wait()
