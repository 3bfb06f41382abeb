"""Steps on host-resident buffers through muon_step_host (pipelined copies in
and out around chunked muon_step calls, on streams the library owns) give
exactly the results of one device-resident muon_step over the whole batch,
for every mix of host and device buffers and every pipeline shape."""
import pytest
import torch

from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl
from muon_newton_schulz_gb300.offload import HostOffloadedMuon

pytestmark = pytest.mark.gpu

ALL = B.MUON_HOST_W | B.MUON_HOST_G | B.MUON_HOST_M


@pytest.mark.parametrize("chunk,slots,host", [
    (1, 2, ALL), (3, 3, ALL), (20, 2, ALL),
    (2, 3, B.MUON_HOST_G),                       # gradient from the host, state on the device
    (4, 2, B.MUON_HOST_W | B.MUON_HOST_M),       # state on the host, gradient on the device
    (3, 4, ALL | B.MUON_HOST_O),                 # and O exported to the host
])
def test_host_buffers_equal_device_resident(chunk, slots, host):
    Ws, Gs, Ms, lrs = wl.make_workload(wl.WORKLOADS["ragged_h384"], "cpu", steady_momentum=True)
    dev = torch.device("cuda", 0)
    Wd, Gd, Md = [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms]
    Od = [torch.empty(w.shape, device=dev) for w in Ws]
    ms = B.MuonStep(0)

    def place(ts, bit):
        return [t.clone().pin_memory() if host & bit else t.to(dev) for t in ts]

    Wh, Gh, Mh = place(Ws, B.MUON_HOST_W), place(Gs, B.MUON_HOST_G), place(Ms, B.MUON_HOST_M)
    Oh = [torch.empty(w.shape).pin_memory() if host & B.MUON_HOST_O else torch.empty(w.shape, device=dev)
          for w in Ws]
    off = HostOffloadedMuon(0, chunk=chunk, slots=slots, host_buffers=host)
    builds = []
    for _ in range(2):
        ms.step(Wd, Gd, Md, lrs, Od)
        off.step(Wh, Gh, Mh, lrs, Oh)
        torch.cuda.synchronize()
        assert off.check_status() == B.MUON_OK
        for i in range(len(Ws)):
            assert torch.equal(Wh[i].cpu().view(torch.int16), Wd[i].cpu().view(torch.int16))
            assert torch.equal(Mh[i].cpu(), Md[i].cpu())
            assert torch.equal(Oh[i].cpu(), Od[i].cpu())
        builds.append(B.muon_plan_builds(off.muon.h))
    # the second step's chunks land in the same slots and reuse their plans
    assert builds[1] == builds[0]
    off.close()
    ms.close()


def test_host_step_time_out_is_reported(monkeypatch):
    """A time-out inside one chunk's step shows in the status word of its slot,
    which muon_check_status on the host-step workspace reads."""
    Ws, Gs, Ms, lrs = wl.make_workload(wl.WORKLOADS["experts_4x256x1024"], "cpu")
    Wh = [w.clone().pin_memory() for w in Ws]
    Gh = [g.clone().pin_memory() for g in Gs]
    Mh = [m.clone().pin_memory() for m in Ms]
    monkeypatch.setenv("MUON_GB300_TEST_WITHHOLD_LOADS", "1")
    off = HostOffloadedMuon(0, chunk=2, slots=2)
    monkeypatch.delenv("MUON_GB300_TEST_WITHHOLD_LOADS")
    off.step(Wh, Gh, Mh, lrs)
    assert off.check_status() == B.MUON_ERR_TIMEOUT
    for a, b in zip(Wh, Ws):
        assert torch.equal(a, b)      # no chunk applied an update
    assert off.check_status() == B.MUON_OK
    off.close()


def test_host_step_with_every_buffer_on_the_device_is_muon_step():
    """host_buffers = 0: nothing is staged or copied; each chunk's step runs on
    the caller's device buffers in place and equals one muon_step."""
    Ws, Gs, Ms, lrs = wl.make_workload(wl.WORKLOADS["odd_shapes"], "cpu", steady_momentum=True)
    dev = torch.device("cuda", 0)
    Wa, Ga, Ma = [w.to(dev) for w in Ws], [g.to(dev) for g in Gs], [m.to(dev) for m in Ms]
    Wb, Mb = [w.to(dev) for w in Ws], [m.to(dev) for m in Ms]
    ms = B.MuonStep(0)
    ms.step(Wa, Ga, Ma, lrs)
    off = HostOffloadedMuon(0, chunk=2, slots=2, host_buffers=0)
    off.step(Wb, Ga, Mb, lrs)
    assert off.check_status() == B.MUON_OK
    for a, b in zip(Wa, Wb):
        assert torch.equal(a, b)
    for a, b in zip(Ma, Mb):
        assert torch.equal(a, b)
    off.close()
    ms.close()
