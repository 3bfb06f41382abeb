"""Host-offloaded steps (state in pinned host memory, pipelined copies and
chunked muon_step calls) give exactly the results of one device-resident
muon_step over the whole batch."""
import pytest
import torch

from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl
from muon_newton_schulz_gb300.offload import HostOffloadedMuon

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chunk,slots", [(1, 2), (3, 3), (20, 2)])
def test_offloaded_equals_device_resident(chunk, slots):
    Ws, Gs, Ms, lrs = wl.make_workload(wl.WORKLOADS["ragged_h384"], "cpu", steady_momentum=True)
    dev = torch.device("cuda", 0)
    Wd, Gd, Md = [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms]
    ms = B.MuonStep(0)
    Wh = [w.clone().pin_memory() for w in Ws]
    Gh = [g.clone().pin_memory() for g in Gs]
    Mh = [m.clone().pin_memory() for m in Ms]
    off = HostOffloadedMuon(0, chunk=chunk, slots=slots)
    for _ in range(2):
        ms.step(Wd, Gd, Md, lrs)
        off.step(Wh, Gh, Mh, lrs)
        torch.cuda.synchronize()
        for i in range(len(Ws)):
            assert torch.equal(Wh[i].view(torch.int16), Wd[i].cpu().view(torch.int16))
            assert torch.equal(Mh[i], Md[i].cpu())
    off.close()
    ms.close()
