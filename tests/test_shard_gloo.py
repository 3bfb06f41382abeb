"""Whole-matrix ownership across ranks (CPU, gloo, world size 2): every
matrix is stepped exactly once, by its owner, with no data exchange; the
gathered results equal a single-process run; the split is balanced."""
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
