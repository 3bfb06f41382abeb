"""Failure detection without a GPU fault: every wait in the tensor-core
kernels is bounded.  A test hook (an environment variable that nothing sets in
normal use, read when a handle is created) makes the first Gram launch of
every step of that handle withhold its loads; its waits then run out after
about a second, the kernel drains, frees its tensor memory and returns,
muon_check_status reports MUON_ERR_TIMEOUT, the step leaves W unchanged, and
the next step on the same context (another handle) is correct again."""
import os

import numpy as np
import pytest
import torch

import oracle.muon_oracle as O
from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_withheld_loads_time_out_and_the_context_survives(monkeypatch):
    Ws, Gs, Ms, lrs = wl.make_workload(wl.WORKLOADS["experts_4x256x1024"], "cpu")
    dev = torch.device("cuda", 0)
    Wd, Gd, Md = [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms]
    monkeypatch.setenv("MUON_GB300_TEST_WITHHOLD_LOADS", "1")
    bad = B.MuonStep(0)
    monkeypatch.delenv("MUON_GB300_TEST_WITHHOLD_LOADS")
    bad.step(Wd, Gd, Md, lrs)
    torch.cuda.synchronize()
    assert bad.check_status() == B.MUON_ERR_TIMEOUT
    assert "bounded wait" in B.muon_last_error_message(bad.h)
    # the last GEMM saw the time-out and left every weight as it was
    for w0, w in zip(Ws, Wd):
        assert torch.equal(w.cpu(), w0)
    assert bad.check_status() == B.MUON_OK   # read and cleared
    bad.close()
    # a fresh step from the original inputs, on a handle without the hook, is correct
    ms = B.MuonStep(0)
    Wd, Gd, Md = [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms]
    Od = [torch.empty(w.shape, device=dev) for w in Ws]
    ms.step(Wd, Gd, Md, lrs, Od)
    torch.cuda.synchronize()
    assert ms.check_status() == B.MUON_OK
    for i in range(len(Ws)):
        res = O.muon_step_matrix(Ws[i].float().numpy(), Gs[i].numpy(), Ms[i].numpy(), lrs[i], O.OracleConfig(),
                                 w_is_bf16=True)
        o = Od[i].cpu().double().numpy()
        assert np.linalg.norm(o - res.O) / np.linalg.norm(res.O) < 2e-2
    ms.close()
