"""Whole-matrix ownership across ranks (CPU, gloo, world size 2): every
matrix is stepped exactly once, by its owner, with no data exchange; the
gathered results equal a single-process run; the split is balanced."""
import io
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.muon_oracle as O
from muon_newton_schulz_gb300 import workloads as wl
from muon_newton_schulz_gb300.shard import owned_indices, owner_partition, rank_loads

SHAPES_WORKLOAD = wl.Workload("tiny_ragged", (
    wl.MatrixSpec(24, 8, 3, "svd", log10_lo=-3.0),
    wl.MatrixSpec(16, 16, 2, "gauss", 1e-3),
    wl.MatrixSpec(8, 40, 4, "gauss", 1.0),
), seed_base=777)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shapes = SHAPES_WORKLOAD.shapes
        mine = owned_indices(shapes, rank, world)
        Ws, Gs, Ms, lrs = wl.make_workload(SHAPES_WORKLOAD, "cpu", indices=set(mine))
        results = {}
        for i, W, G, M, lr in zip(mine, Ws, Gs, Ms, lrs):
            res = O.muon_step_matrix(W.float().numpy(), G.numpy(), M.numpy(), lr, O.OracleConfig(), w_is_bf16=True)
            results[i] = (res.W, res.M)
        gathered = [None] * world
        dist.all_gather_object(gathered, results)   # only to check, not part of the step
        if rank == 0:
            merged = {}
            for part in gathered:
                assert not (set(part) & set(merged)), "a matrix was stepped twice"
                merged.update(part)
            out.put(sorted(merged.items()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_step_each_matrix_once_and_match_single_process():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    merged = out.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    n = SHAPES_WORKLOAD.n_matrices
    assert [i for i, _ in merged] == list(range(n))
    Ws, Gs, Ms, lrs = wl.make_workload(SHAPES_WORKLOAD, "cpu")
    for (i, (W1, M1)), W, G, M, lr in zip(merged, Ws, Gs, Ms, lrs):
        res = O.muon_step_matrix(W.float().numpy(), G.numpy(), M.numpy(), lr, O.OracleConfig(), w_is_bf16=True)
        assert np.array_equal(res.W, W1) and np.array_equal(res.M, M1)


def test_partition_is_deterministic_and_balanced():
    shapes = wl.WORKLOADS["ragged_h6144"].shapes
    for world in (1, 2, 3, 4, 8):
        own = owner_partition(shapes, world)
        assert own == owner_partition(shapes, world)
        assert sorted(set(own)) == list(range(min(world, len(shapes))))
        loads = rank_loads(shapes, world)
        biggest = max(wl.symmetric_flops(r, c) for r, c in shapes)
        # LPT bound: no rank exceeds the mean load by more than one matrix
        assert max(loads) <= sum(loads) / world + biggest
    # identical matrices split evenly
    own = owner_partition([(2048, 8192)] * 16, 4)
    assert [own.count(k) for k in range(4)] == [4, 4, 4, 4]


def test_empty_matrices_cost_nothing():
    own = owner_partition([(0, 5), (8, 8), (3, 0)], 2)
    assert len(own) == 3


# --- FlexShard: dense matrices row-sharded and gathered to their owner ------------

FLEX_WORKLOAD = wl.Workload("tiny_flexshard", (
    wl.MatrixSpec(24, 8, 3, "svd", log10_lo=-3.0),    # experts (tall)
    wl.MatrixSpec(8, 40, 2, "gauss", 1.0),            # experts (wide)
    wl.MatrixSpec(17, 30, 2, "gauss", 1e-3),          # dense, rows not divisible by the world size
    wl.MatrixSpec(33, 12, 1, "svd", log10_lo=-4.0),   # dense, tall
    wl.MatrixSpec(1, 16, 1, "gauss", 1.0),            # dense with one row: a rank holds an empty shard
), seed_base=4242)
FLEX_DENSE = [False] * 5 + [True] * 4


def _oracle_step_fn(calls):
    """In-place step of whole matrices with the fp64 oracle (the library's
    MuonStep.step plays this part on a GPU)."""
    def step(Ws, Gs, Ms, lrs):
        for W, G, M, lr in zip(Ws, Gs, Ms, lrs):
            calls.append(tuple(W.shape))
            res = O.muon_step_matrix(W.float().numpy(), G.numpy(), M.numpy(), lr, O.OracleConfig(),
                                     w_is_bf16=(W.dtype == torch.bfloat16))
            W.copy_(torch.from_numpy(res.W).to(W.dtype))
            M.copy_(torch.from_numpy(res.M))
    return step


def _flex_worker(rank, world, port, out, steps):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from muon_newton_schulz_gb300.shard import FlexShardPlan, FlexShardStep
        plan = FlexShardPlan.build(FLEX_WORKLOAD.shapes, FLEX_DENSE, world)
        Ws, Gs, Ms, lrs = wl.make_workload(FLEX_WORKLOAD, "cpu", steady_momentum=True)
        local = {}
        for i in range(len(Ws)):
            if plan.dense[i]:
                b, e = plan.shards[i][rank]
                local[i] = (Ws[i][b:e].clone(), Gs[i][b:e].clone(), Ms[i][b:e].clone())
            elif plan.owner[i] == rank:
                local[i] = (Ws[i].clone(), Gs[i].clone(), Ms[i].clone())
        calls = []
        runner = FlexShardStep(plan, rank, _oracle_step_fn(calls), lambda shape, dt: torch.empty(shape, dtype=dt))
        for s in range(steps):
            # a new gradient each step, the same on every rank (shards of it)
            G_step = {i: (local[i][1] * (1.0 + s)) for i in local}
            runner.step({i: (local[i][0], G_step[i], local[i][2]) for i in local}, lrs)
        # by value: tensors sent through the queue would live in this
        # process's shared memory, which is gone once it exits
        buf = io.BytesIO()
        torch.save({i: (local[i][0], local[i][2]) for i in local}, buf)
        out.put((rank, buf.getvalue(), calls))
    finally:
        dist.destroy_process_group()


def test_flexshard_two_ranks_equal_single_process():
    from muon_newton_schulz_gb300.shard import FlexShardPlan
    world, steps = 2, 2
    plan = FlexShardPlan.build(FLEX_WORKLOAD.shapes, FLEX_DENSE, world)
    assert any(plan.owner[i] == 0 for i in range(9)) and any(plan.owner[i] == 1 for i in range(9))
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_flex_worker, args=(r, world, port, out, steps)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict((r, (torch.load(io.BytesIO(loc)), calls)) for r, loc, calls in (out.get(timeout=180) for _ in range(world)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # single process: every matrix whole, the same gradients
    Ws, Gs, Ms, lrs = wl.make_workload(FLEX_WORKLOAD, "cpu", steady_momentum=True)
    ref_calls = []
    step = _oracle_step_fn(ref_calls)
    for s in range(steps):
        step(Ws, [g * (1.0 + s) for g in Gs], Ms, lrs)
    n = len(Ws)
    # every matrix stepped exactly once per step, by its owner, whole
    all_calls = sorted(got[0][1] + got[1][1])
    assert all_calls == sorted(ref_calls)
    for i in range(n):
        if plan.dense[i]:
            parts = [got[k][0][i] for k in range(world)]
            W = torch.cat([p[0] for p in parts])
            M = torch.cat([p[1] for p in parts])
        else:
            W, M = got[plan.owner[i]][0][i]
            assert i not in got[1 - plan.owner[i]][0]    # the other rank never held it
        assert torch.equal(W, Ws[i]) and torch.equal(M, Ms[i]), i


def test_flexshard_plan_shards_and_traffic():
    from muon_newton_schulz_gb300.shard import FlexShardPlan, row_shards
    assert row_shards(17, 2) == [(0, 9), (9, 17)]
    assert row_shards(1, 3) == [(0, 1), (1, 1), (1, 1)]
    for world in (1, 2, 3, 8):
        for rows in (1, 7, 64, 6144):
            sh = row_shards(rows, world)
            assert sh[0][0] == 0 and sh[-1][1] == rows
            assert all(a[1] == b[0] for a, b in zip(sh, sh[1:]))
            assert max(e - b for b, e in sh) - min(e - b for b, e in sh) <= 1
    # the pages' mixed layer at hidden 6144: experts owned whole, projections sharded
    w = wl.WORKLOADS["ragged_h6144"]
    dense = [s.rows == s.cols for s in w.specs for _ in range(s.count)]
    plan = FlexShardPlan.build(w.shapes, dense, 4)
    for rank in range(4):
        for i in plan.experts_of(rank):
            assert plan.local_shape(i, rank) == w.shapes[i]
            assert all(plan.local_shape(i, k) is None for k in range(4) if k != rank)
    # four 6144^2 projections, each 3/4 away from its owner, bf16 W
    assert plan.bytes_moved() == 4 * (6144 * 6144 * 3 // 4) * (4 + 4 + 2 + 2 + 4)
    assert FlexShardPlan.build(w.shapes, dense, 1).bytes_moved() == 0
