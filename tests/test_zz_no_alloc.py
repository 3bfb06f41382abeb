"""muon_step_noalloc, the entry point for callers that may not allocate
device memory (runtimes that reserve all memory up front, plugins confined to
a host framework's tensors): it runs the same step on the library's fixed
device array instead of a caller workspace.  The kernels and their schedule
do not depend on where the workspace lives, so W, M and O must equal
muon_step's bit for bit, on two consecutive steps.  A bounded-wait time-out
under this entry point is reported through muon_check_status(h, NULL, s),
which reads the status word inside the fixed array.  Kept in a file of its
own that pytest collects last."""
import pytest
import torch

from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _device_inputs(name, indices=None):
    dev = torch.device("cuda", 0)
    Ws, Gs, Ms, lrs = wl.make_workload(wl.WORKLOADS[name], "cpu", steady_momentum=True, indices=indices)
    return [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms], lrs


def _clone(ts):
    return [t.clone() for t in ts]


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_noalloc_matches_muon_step_on_two_steps(mode):
    Ws, Gs, Ms, lrs = _device_inputs("ragged_h384")
    Wa, Ma = _clone(Ws), _clone(Ms)     # driven by muon_step
    Wb, Mb = _clone(Ws), _clone(Ms)     # driven by muon_step_noalloc
    Oa = [torch.empty(w.shape, device=w.device) for w in Ws]
    Ob = [torch.empty(w.shape, device=w.device) for w in Ws]
    ref = B.MuonStep(0, mode=mode)
    h = B.MuonStep(0, mode=mode)
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):
        G = [g * (1.0 + step) for g in Gs]
        ref.step(Wa, G, Ma, lrs, Oa)
        descs, n = B.MuonStep.descs_from_tensors(Wb, G, Mb, lrs, Ob)
        assert h.workspace_bytes(descs, n) <= B.MUON_STATIC_WORKSPACE_BYTES
        st = B.muon_step_noalloc(h.h, descs, n, stream)
        assert st == B.MUON_OK, B.muon_last_error_message(h.h)
        torch.cuda.synchronize()
        assert B.muon_check_status(h.h, None, stream) == B.MUON_OK
        for i in range(len(Ws)):
            assert torch.equal(Ob[i], Oa[i]), (step, i)
            assert torch.equal(Mb[i], Ma[i]), (step, i)
            assert torch.equal(Wb[i], Wa[i]), (step, i)
    ref.close()
    h.close()


def test_noalloc_time_out_is_reported(monkeypatch):
    """The load-withholding test hook (read when a handle is created) makes the
    step's first Gram launch give up its bounded waits; the status word in the
    fixed array then reads MUON_ERR_TIMEOUT, W is left as it was, and the next
    call on a handle without the hook is correct."""
    Ws, Gs, Ms, lrs = _device_inputs("experts_4x256x1024")
    W0 = _clone(Ws)
    monkeypatch.setenv("MUON_GB300_TEST_WITHHOLD_LOADS", "1")
    bad = B.MuonStep(0)
    monkeypatch.delenv("MUON_GB300_TEST_WITHHOLD_LOADS")
    stream = torch.cuda.current_stream().cuda_stream
    descs, n = B.MuonStep.descs_from_tensors(Ws, Gs, _clone(Ms), lrs)
    assert B.muon_step_noalloc(bad.h, descs, n, stream) == B.MUON_OK
    torch.cuda.synchronize()
    assert B.muon_check_status(bad.h, None, stream) == B.MUON_ERR_TIMEOUT
    assert "bounded wait" in B.muon_last_error_message(bad.h)
    for a, b in zip(Ws, W0):
        assert torch.equal(a, b)
    assert B.muon_check_status(bad.h, None, stream) == B.MUON_OK   # read and cleared
    bad.close()
    # the fixed array is usable again: a normal call equals muon_step
    good = B.MuonStep(0)
    ref = B.MuonStep(0)
    Wa, Ma, Wb, Mb = _clone(W0), _clone(Ms), _clone(W0), _clone(Ms)
    ref.step(Wa, Gs, Ma, lrs)
    descs, n = B.MuonStep.descs_from_tensors(Wb, Gs, Mb, lrs)
    assert B.muon_step_noalloc(good.h, descs, n, stream) == B.MUON_OK
    torch.cuda.synchronize()
    assert B.muon_check_status(good.h, None, stream) == B.MUON_OK
    for i in range(len(Wa)):
        assert torch.equal(Wa[i], Wb[i]) and torch.equal(Ma[i], Mb[i])
    good.close()
    ref.close()


def test_noalloc_rejects_batches_beyond_the_fixed_array():
    # one 2048 x 4096 matrix needs about 98 MiB of workspace
    dev = torch.device("cuda", 0)
    W = torch.zeros(2048, 4096, dtype=torch.bfloat16, device=dev)
    G = torch.randn(2048, 4096, device=dev)
    M = torch.zeros_like(G)
    h = B.MuonStep(0)
    descs, n = B.MuonStep.descs_from_tensors([W], [G], [M], [1e-3])
    assert h.workspace_bytes(descs, n) > B.MUON_STATIC_WORKSPACE_BYTES
    W0 = W.clone()
    st = B.muon_step_noalloc(h.h, descs, n, torch.cuda.current_stream().cuda_stream)
    assert st == B.MUON_ERR_WORKSPACE
    assert "MUON_STATIC_WORKSPACE_BYTES" in B.muon_last_error_message(h.h)
    torch.cuda.synchronize()
    assert torch.equal(W, W0) and torch.count_nonzero(M) == 0
    # an empty batch is accepted and launches nothing
    arr, _ = B.make_descs([])
    assert B.muon_step_noalloc(h.h, arr, 0, 0) == B.MUON_OK
    h.close()
