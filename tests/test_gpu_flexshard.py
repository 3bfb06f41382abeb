"""FlexShardStep on one GPU with the library's step: at world size 1 every
dense matrix is one whole shard, gathered into the owner's buffer, stepped by
muon_step and copied back; experts are stepped in place.  The result equals
one muon_step over the batch bit for bit.  (The exchange between ranks is
tested on CPU with gloo in test_shard_gloo.py; every run here has one GPU.)"""
import pytest
import torch

from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl
from muon_newton_schulz_gb300.shard import FlexShardPlan, FlexShardStep

pytestmark = pytest.mark.gpu


def test_flexshard_single_rank_equals_muon_step():
    w = wl.WORKLOADS["ragged_h384"]
    dense = [s.rows == s.cols for s in w.specs for _ in range(s.count)]
    Ws, Gs, Ms, lrs = wl.make_workload(w, "cpu", steady_momentum=True)
    dev = torch.device("cuda", 0)
    Wa, Ga, Ma = [x.to(dev) for x in Ws], [x.to(dev) for x in Gs], [x.to(dev) for x in Ms]
    ref = B.MuonStep(0)
    ref.step(Wa, Ga, Ma, lrs)
    plan = FlexShardPlan.build(w.shapes, dense, 1)
    ms = B.MuonStep(0)
    runner = FlexShardStep(plan, 0, ms.step, lambda shape, dt: torch.empty(shape, dtype=dt, device=dev))
    local = {i: (Ws[i].to(dev), Gs[i].to(dev), Ms[i].to(dev)) for i in range(len(Ws))}
    runner.step(local, lrs)
    torch.cuda.synchronize()
    assert ms.check_status() == B.MUON_OK
    for i in range(len(Ws)):
        assert torch.equal(local[i][0], Wa[i]) and torch.equal(local[i][2], Ma[i]), i
    ms.close()
    ref.close()
