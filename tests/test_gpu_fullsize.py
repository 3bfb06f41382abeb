"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (the whole batch in one muon_step call, bf16 mode): the oracle checks
sampled matrices one by one, and properties that hold at any size are checked
on every matrix."""
import numpy as np
import pytest
import torch

import oracle.muon_oracle as O
from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl
from gpu_helpers import check_matrix, rel_frob

pytestmark = pytest.mark.gpu


def _run_full(name, samples, steady=False):
    """Whole workload generated on the GPU and stepped in one call; returns
    host copies of the inputs and outputs of the sampled matrices, plus the
    per-matrix norms of O for every matrix."""
    w = wl.WORKLOADS[name]
    dev = torch.device("cuda", 0)
    Ws, Gs, Ms, lrs = wl.make_workload(w, dev, steady_momentum=steady)
    W0 = {i: Ws[i].cpu() for i in samples}
    G0 = {i: Gs[i].cpu() for i in samples}
    M0 = {i: Ms[i].cpu() for i in samples}
    Os = [torch.empty(x.shape, dtype=torch.float32, device=dev) for x in Ws]
    ms = B.MuonStep(0)
    ms.step(Ws, Gs, Ms, lrs, Os)
    torch.cuda.synchronize()
    assert ms.check_status() == B.MUON_OK
    ms.close()
    # O has singular values p^5(sigma) in about [0.47, 1.2] on its support:
    # every matrix's ||O||_F^2 / min(r, c) must lie in that band and be finite
    for i, o in enumerate(Os):
        q = float((o.double() ** 2).sum() / min(o.shape))
        assert np.isfinite(q) and 0.05 < q < 1.5, (i, q)
    out = {i: (Ws[i].cpu(), Ms[i].cpu(), Os[i].cpu()) for i in samples}
    return W0, G0, M0, lrs, out


def _check_samples(name, samples, tol=2e-2, steady=False):
    W0, G0, M0, lrs, out = _run_full(name, samples, steady)
    errs = []
    for i in samples:
        res = O.muon_step_matrix(W0[i].float().numpy(), G0[i].numpy(), M0[i].numpy(), lrs[i],
                                 O.OracleConfig(), w_is_bf16=(W0[i].dtype == torch.bfloat16))
        Wg, Mg, Og = out[i]
        errs.append(check_matrix(W0[i], G0[i], M0[i], lrs[i], Wg, Mg, Og, res, tol, f"{name}[{i}]"))
    print(f"\nERR {name} samples={sorted(samples)} max_rel_err={max(errs):.3e}")
    return errs


def test_experts_16x2048x8192_sampled():
    _check_samples("experts_16x2048x8192", {0, 15}, steady=True)


def test_dense_7680x7680():
    _check_samples("dense_7680x7680", {0})


def test_ragged_h6144_sampled():
    # one matrix of each shape: tall 6144x2048, square 6144^2, wide 2048x6144
    _check_samples("ragged_h6144", {0, 32, 40})


def test_single_256x512_full():
    _check_samples("single_256x512", {0})


def test_experts_128x2048x8192_sampled():
    _check_samples("experts_128x2048x8192", {0, 127})


def test_mlp_and_qproj_shapes():
    # 3072 x 12288 (wide) and 2048 x 1024 (tall) in one ragged batch
    _check_samples("mlp_and_qproj", {0, 1, 4})
