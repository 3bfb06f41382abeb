"""Properties of the CUDA path that hold at any size: bitwise determinism,
independence from batch composition and order, multi-step momentum and
resume, non-finite isolation, degenerate inputs, launch counts, profiling."""
import numpy as np
import pytest
import torch

import oracle.muon_oracle as O
from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl
from gpu_helpers import check_matrix, oracle_for, run_gpu

pytestmark = pytest.mark.gpu


def _inputs(name, steady=False, indices=None):
    return wl.make_workload(wl.WORKLOADS[name], "cpu", steady_momentum=steady, indices=indices)


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_bitwise_deterministic(mode):
    Ws, Gs, Ms, lrs = _inputs("ragged_h384", steady=True)
    a = run_gpu(Ws, Gs, Ms, lrs, mode=mode)
    b = run_gpu(Ws, Gs, Ms, lrs, mode=mode)
    for x, y in zip(a, b):
        for u, v in zip(x, y):
            assert torch.equal(u.view(torch.int16) if u.dtype == torch.bfloat16 else u.view(torch.int32),
                               v.view(torch.int16) if v.dtype == torch.bfloat16 else v.view(torch.int32))


def test_batch_composition_and_order_do_not_matter():
    Ws, Gs, Ms, lrs = _inputs("ragged_h384", steady=True)
    full = run_gpu(Ws, Gs, Ms, lrs)
    for i in (0, 7, 10):
        alone = run_gpu([Ws[i]], [Gs[i]], [Ms[i]], [lrs[i]])
        assert torch.equal(alone[2][0], full[2][i])
        assert torch.equal(alone[0][0].float(), full[0][i].float())
    rev = list(reversed(range(len(Ws))))
    back = run_gpu([Ws[i] for i in rev], [Gs[i] for i in rev], [Ms[i] for i in rev], [lrs[i] for i in rev])
    for k, i in enumerate(rev):
        assert torch.equal(back[2][k], full[2][i])
        assert torch.equal(back[1][k], full[1][i])


def test_multistep_and_resume():
    Ws, Gs, Ms, lrs = _inputs("experts_4x256x1024")
    dev = torch.device("cuda", 0)
    Wd = [w.to(dev) for w in Ws]
    Md = [m.to(dev) for m in Ms]
    Od = [torch.empty(w.shape, dtype=torch.float32, device=dev) for w in Ws]
    ms = B.MuonStep(0)
    rng = torch.Generator().manual_seed(123)
    saved = None
    for step in range(3):
        G = [torch.randn(w.shape, generator=rng) * 1e-3 for w in Ws]
        W_before = [w.cpu() for w in Wd]
        M_before = [m.cpu() for m in Md]
        if step == 2:
            saved = ([w.clone() for w in Wd], [m.clone() for m in Md], [g.clone() for g in G])
        ms.step(Wd, [g.to(dev) for g in G], Md, lrs, Od)
        torch.cuda.synchronize()
        for i in range(len(Ws)):
            res = oracle_for(W_before[i], G[i], M_before[i], lrs[i])
            check_matrix(W_before[i], G[i], M_before[i], lrs[i], Wd[i].cpu(), Md[i].cpu(), Od[i].cpu(), res, 2e-2)
    # resume from the checkpoint of step 2: bit-identical
    W3 = [w.cpu() for w in Wd]
    M3 = [m.cpu() for m in Md]
    Wr, Mr, Gr = saved
    ms.step(Wr, [g.to(dev) for g in Gr], Mr, lrs)
    torch.cuda.synchronize()
    for i in range(len(Ws)):
        assert torch.equal(Wr[i].cpu().view(torch.int16), W3[i].view(torch.int16))
        assert torch.equal(Mr[i].cpu(), M3[i])
    ms.close()


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_nonfinite_stays_in_its_matrix(mode):
    Ws, Gs, Ms, lrs = _inputs("experts_4x256x1024")
    clean = run_gpu(Ws, Gs, Ms, lrs, mode=mode)
    Gbad = [g.clone() for g in Gs]
    Gbad[1][5, 7] = float("nan")
    dirty = run_gpu(Ws, Gbad, Ms, lrs, mode=mode)
    assert torch.isnan(dirty[1][1][5, 7])
    assert torch.isnan(dirty[2][1]).all()
    for i in (0, 2, 3):
        assert torch.equal(dirty[2][i], clean[2][i])
        assert torch.equal(dirty[0][i].float(), clean[0][i].float())


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_zero_gradient_leaves_weights(mode):
    Ws, Gs, Ms, lrs = _inputs("odd_shapes")
    Z = [torch.zeros_like(g) for g in Gs]
    W, M, Oo = run_gpu(Ws, Z, [torch.zeros_like(m) for m in Ms], lrs, mode=mode)
    for i in range(len(Ws)):
        assert torch.count_nonzero(Oo[i]) == 0
        assert torch.equal(W[i].float(), Ws[i].float())
        assert torch.count_nonzero(M[i]) == 0


def test_empty_matrices_are_skipped():
    Ws, Gs, Ms, lrs = _inputs("odd_shapes", indices={0, 3})
    e = torch.zeros(0, 7)
    W, M, Oo = run_gpu([Ws[0], e.to(torch.bfloat16), Ws[1]], [Gs[0], e, Gs[1]], [Ms[0], e, Ms[1]],
                       [lrs[0], 1.0, lrs[1]])
    ref = run_gpu([Ws[0], Ws[1]], [Gs[0], Gs[1]], [Ms[0], Ms[1]], [lrs[0], lrs[1]])
    assert torch.equal(Oo[0], ref[2][0]) and torch.equal(Oo[2], ref[2][1])


def test_strided_inputs():
    """Leading dimensions larger than cols (row padding) on every buffer."""
    Ws, Gs, Ms, lrs = _inputs("odd_shapes", indices={0, 1})
    dev = torch.device("cuda", 0)
    pads = []
    for W, G, M in zip(Ws, Gs, Ms):
        r, c = W.shape
        Wp = torch.zeros(r, c + 8, dtype=W.dtype, device=dev)[:, :c]
        Gp = torch.zeros(r, c + 4, device=dev)[:, :c]
        Mp = torch.zeros(r, c + 12, device=dev)[:, :c]
        Wp.copy_(W)
        Gp.copy_(G)
        Mp.copy_(M)
        pads.append((Wp, Gp, Mp))
    ms = B.MuonStep(0)
    Od = [torch.empty(w.shape, device=dev) for w in Ws]
    ms.step([p[0] for p in pads], [p[1] for p in pads], [p[2] for p in pads], lrs, Od)
    torch.cuda.synchronize()
    ref = run_gpu(Ws, Gs, Ms, lrs)
    for i in range(2):
        assert torch.equal(Od[i].cpu(), ref[2][i])
        assert torch.equal(pads[i][0].cpu().float(), ref[0][i].float())
    ms.close()


@pytest.mark.parametrize("iters", [0, 5])
def test_launch_count_and_profile(iters):
    Ws, Gs, Ms, lrs = _inputs("ragged_h384")
    dev = torch.device("cuda", 0)
    ms = B.MuonStep(0, ns_iters=iters)
    Wd, Gd, Md = [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms]
    assert B.muon_set_profiling(ms.h, True) == B.MUON_OK
    n0 = B.muon_launch_count(ms.h)
    ms.step(Wd, Gd, Md, lrs)
    ms.step(Wd, Gd, Md, lrs)
    # tensor-core mode folds the weight update into the last GEMM; with zero
    # iterations a separate apply kernel runs
    apply_launches = 0 if iters > 0 else 1
    assert B.muon_launch_count(ms.h) - n0 == 2 * (2 + 3 * iters + apply_launches)
    st, prof = B.muon_read_profile(ms.h)
    assert st == B.MUON_OK and prof.steps == 2
    assert prof.launches[0] == 4 and prof.launches[4] == 2 * apply_launches
    if iters:
        assert prof.launches[3] == 2 * iters and prof.ms[3] > 0
    ms.close()


def test_rank_deficient_gradient():
    """A rank-3 gradient keeps rank 3 after the step (within bf16 noise)."""
    g = torch.Generator().manual_seed(5)
    G = (torch.randint(-4, 5, (200, 3), generator=g).float() @ torch.randint(-4, 5, (3, 520), generator=g).float())
    W = torch.zeros(200, 520, dtype=torch.bfloat16)
    _, _, Oo = run_gpu([W], [G], [torch.zeros_like(G)], [1e-3])
    s = np.linalg.svd(Oo[0].double().numpy(), compute_uv=False)
    assert s[2] > 0.1 and s[3] < 1e-2 * s[0]
    res = oracle_for(W, G, torch.zeros_like(G), 1e-3)
    assert np.linalg.norm(Oo[0].numpy() - res.O) / np.linalg.norm(res.O) < 2e-2


def test_workspace_errors_leave_state_untouched():
    """NULL, misaligned or short workspaces are refused before any launch:
    MUON_ERR_WORKSPACE with a message, W and M unchanged; the exact size runs."""
    Ws, Gs, Ms, lrs = _inputs("experts_4x256x1024", steady=True)
    dev = torch.device("cuda", 0)
    Wd, Gd, Md = [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms]
    ms = B.MuonStep(0)
    descs, n = ms.descs_from_tensors(Wd, Gd, Md, lrs)
    need = ms.workspace_bytes(descs, n)
    ws = torch.empty(need + 512, dtype=torch.uint8, device=dev)
    base = ws.data_ptr()
    assert base % 256 == 0
    s = torch.cuda.current_stream(dev).cuda_stream
    for ptr, nbytes, msg in ((0, need, "NULL"), (base + 16, need, "256-byte aligned"), (base, need - 1, "too small")):
        assert B.muon_step(ms.h, descs, n, ptr, nbytes, s) == B.MUON_ERR_WORKSPACE
        assert msg in B.muon_last_error_message(ms.h)
    torch.cuda.synchronize(dev)
    for i in range(len(Ws)):
        assert torch.equal(Wd[i].cpu().view(torch.int16), Ws[i].view(torch.int16))
        assert torch.equal(Md[i].cpu(), Ms[i])
    assert B.muon_step(ms.h, descs, n, base, need, s) == B.MUON_OK
    torch.cuda.synchronize(dev)
    assert B.muon_check_status(ms.h, base, s) == B.MUON_OK
    ms.close()


def _device_copies(batch, dev):
    Ws, Gs, Ms, lrs = batch
    return ([w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms], lrs,
            [torch.empty(w.shape, dtype=torch.float32, device=dev) for w in Ws])


def _assert_same(dev_out, ref):
    Wd, _, Md, _, Od = dev_out
    for i in range(len(Wd)):
        assert torch.equal(Wd[i].cpu().float(), ref[0][i].float())
        assert torch.equal(Md[i].cpu(), ref[1][i])
        assert torch.equal(Od[i].cpu(), ref[2][i])


def test_one_handle_many_batches_and_streams():
    """One handle steps differently shaped batches in turn on a side stream,
    and two handles step on two streams at once: every result equals a fresh
    handle's on the default stream, bit for bit."""
    dev = torch.device("cuda", 0)
    A = _inputs("experts_4x256x1024", steady=True)
    Bt = _inputs("odd_shapes", steady=True)
    ref_a, ref_b = run_gpu(*A), run_gpu(*Bt)
    side = torch.cuda.Stream(dev)
    ms = B.MuonStep(0)
    for batch, ref in ((A, ref_a), (Bt, ref_b), (A, ref_a)):
        d = _device_copies(batch, dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            ms.step(d[0], d[1], d[2], d[3], d[4], stream=side.cuda_stream)
        side.synchronize()
        assert ms.check_status(stream=side.cuda_stream) == B.MUON_OK
        _assert_same(d, ref)
    ms.close()
    h1, h2 = B.MuonStep(0), B.MuonStep(0)
    da, db = _device_copies(A, dev), _device_copies(Bt, dev)
    for h, d in ((h1, da), (h2, db)):
        descs, n = h.descs_from_tensors(d[0], d[1], d[2], d[3], d[4])
        h.workspace(h.workspace_bytes(descs, n))
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s1):
        h1.step(da[0], da[1], da[2], da[3], da[4], stream=s1.cuda_stream)
    with torch.cuda.stream(s2):
        h2.step(db[0], db[1], db[2], db[3], db[4], stream=s2.cuda_stream)
    torch.cuda.synchronize(dev)
    assert h1.check_status(stream=s1.cuda_stream) == B.MUON_OK
    assert h2.check_status(stream=s2.cuda_stream) == B.MUON_OK
    _assert_same(da, ref_a)
    _assert_same(db, ref_b)
    h1.close()
    h2.close()


def test_repeated_batch_reuses_its_plan():
    """A batch stepped again with the same descriptors and workspace reuses the
    handle's cached plan (no new validation, tile lists or tensor maps) and
    gives exactly what a handle building the plan from scratch gives; a changed
    descriptor (here the learning rate) builds a new plan."""
    Ws, Gs, Ms, lrs = _inputs("ragged_h384", steady=True)
    dev = torch.device("cuda", 0)
    Wa, Ma = [w.to(dev) for w in Ws], [m.to(dev) for m in Ms]
    Gd = [g.to(dev) for g in Gs]
    cached = B.MuonStep(0)
    descs, n = cached.descs_from_tensors(Wa, Gd, Ma, lrs)
    for _ in range(3):
        cached.step_descs(descs, n)
    assert B.muon_plan_builds(cached.h) == 1
    assert B.muon_graph_launches(cached.h) == 2   # the first step of a plan runs eagerly
    Wb, Mb = [w.to(dev) for w in Ws], [m.to(dev) for m in Ms]
    for _ in range(3):
        fresh = B.MuonStep(0)       # a new handle plans from scratch every step
        fresh.step(Wb, Gd, Mb, lrs)
        torch.cuda.synchronize()
        assert B.muon_plan_builds(fresh.h) == 1
        fresh.close()
    torch.cuda.synchronize()
    assert cached.check_status() == B.MUON_OK
    for a, b in zip(Wa, Wb):
        assert torch.equal(a, b)
    for a, b in zip(Ma, Mb):
        assert torch.equal(a, b)
    descs2, n2 = cached.descs_from_tensors(Wa, Gd, Ma, [2 * x for x in lrs])
    cached.step_descs(descs2, n2)
    assert B.muon_plan_builds(cached.h) == 2
    cached.step_descs(descs, n)       # the first batch is still cached
    assert B.muon_plan_builds(cached.h) == 2
    torch.cuda.synchronize()
    cached.close()


def test_cached_plan_replays_as_a_graph():
    """From a cached plan's second step on, the handle replays the step as a
    CUDA graph it captured once; replays equal eager steps bit for bit, on any
    stream, and profiling switches back to launching the kernels one by one."""
    Ws, Gs, Ms, lrs = _inputs("ragged_h384", steady=True)
    dev = torch.device("cuda", 0)
    Gd = [g.to(dev) for g in Gs]
    Wa, Ma = [w.to(dev) for w in Ws], [m.to(dev) for m in Ms]   # replayed
    Wb, Mb = [w.to(dev) for w in Ws], [m.to(dev) for m in Ms]   # eager (profiling on)
    rep = B.MuonStep(0)
    eager = B.MuonStep(0)
    assert B.muon_set_profiling(eager.h, True) == B.MUON_OK
    d_rep, n = rep.descs_from_tensors(Wa, Gd, Ma, lrs)
    d_eag, _ = eager.descs_from_tensors(Wb, Gd, Mb, lrs)
    side = torch.cuda.Stream(dev)
    per_step = None
    for k in range(4):
        before = B.muon_launch_count(rep.h)
        if k == 2:
            with torch.cuda.stream(side):
                rep.step_descs(d_rep, n, stream=side.cuda_stream)
            torch.cuda.current_stream(dev).wait_stream(side)
        else:
            rep.step_descs(d_rep, n)
        eager.step_descs(d_eag, n)
        per_step = per_step or B.muon_launch_count(rep.h) - before
        assert B.muon_launch_count(rep.h) - before == per_step
    torch.cuda.synchronize()
    assert B.muon_graph_launches(rep.h) == 3 and B.muon_graph_launches(eager.h) == 0
    assert rep.check_status() == B.MUON_OK and eager.check_status() == B.MUON_OK
    for a, b in zip(Wa, Wb):
        assert torch.equal(a, b)
    for a, b in zip(Ma, Mb):
        assert torch.equal(a, b)
    st, prof = B.muon_read_profile(eager.h)
    assert st == B.MUON_OK and prof.steps == 4
    rep.close()
    eager.close()
