"""muon_step_noalloc, the entry point for callers that may not allocate
device memory (runtimes that reserve all memory up front, plugins confined to
a host framework's tensors): it runs the same step on the library's fixed
device array instead of a caller workspace.  Checked against muon_step on
two consecutive steps, and for its size limit.  Kept in a file of its own that
pytest collects last."""
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
        tol = 2e-2 if mode == B.MUON_MODE_BF16 else 1e-4
        for i in range(len(Ws)):
            rel = (Ob[i] - Oa[i]).norm() / Oa[i].norm()
            assert rel <= tol
            assert torch.equal(Mb[i], Ma[i])
            assert (Wb[i].float() - Wa[i].float()).abs().max() <= 1e-2 * Wa[i].float().abs().max()
    ref.close()
    h.close()


def test_noalloc_rejects_batches_beyond_the_fixed_array():
    Ws, Gs, Ms, lrs = _device_inputs("experts_4x256x1024", indices={0})
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
