"""Failure detection without a GPU fault: every wait in the tensor-core
kernels is bounded.  A test hook (an environment variable that nothing sets in
normal use) makes the first Gram launch of a step withhold its loads; its
waits then run out after about a second, the kernel drains, frees its tensor
memory and returns, muon_check_status reports MUON_ERR_TIMEOUT, and the next
step on the same context is correct again."""
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
    ms = B.MuonStep(0)
    Wd, Gd, Md = [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms]
    monkeypatch.setenv("MUON_GB300_TEST_WITHHOLD_LOADS", "1")
    ms.step(Wd, Gd, Md, lrs)
    torch.cuda.synchronize()
    assert ms.check_status() == B.MUON_ERR_TIMEOUT
    assert "bounded wait" in B.muon_last_error_message(ms.h)
    monkeypatch.delenv("MUON_GB300_TEST_WITHHOLD_LOADS")
    # the status word was read and cleared; a fresh step from the original
    # inputs is correct
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
