"""muon_step issues only kernel launches on the caller's stream (no host
synchronisation, allocation or copy), so a step can be captured in a CUDA
graph and replayed: replays give bitwise the results of eager steps, and the
first replay matches the fp64 oracle like any step."""
import numpy as np
import pytest
import torch

from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl
from gpu_helpers import check_matrix, oracle_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["single_256x512", "ragged_h384"])
def test_graph_replay_equals_eager(name):
    dev = torch.device("cuda", 0)
    Ws, Gs, Ms, lrs = wl.make_workload(wl.WORKLOADS[name], dev, steady_momentum=True)
    We, Me = [w.clone() for w in Ws], [m.clone() for m in Ms]
    Wg, Mg = [w.clone() for w in Ws], [m.clone() for m in Ms]
    eager = B.MuonStep(0)
    graphed = B.MuonStep(0)
    descs, n = graphed.descs_from_tensors(Wg, Gs, Mg, lrs)
    ws = graphed.workspace(graphed.workspace_bytes(descs, n))
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        st = B.muon_step(graphed.h, descs, n, ws.data_ptr(), ws.numel(), side.cuda_stream)
    assert st == B.MUON_OK
    torch.cuda.synchronize()
    W0 = [w.cpu() for w in Wg]
    M0 = [m.cpu() for m in Mg]
    for rep in range(3):
        eager.step(We, Gs, Me, lrs)
        graph.replay()
        torch.cuda.synchronize()
        if rep == 0:
            # the captured step against the oracle: W from the graph, O from
            # the bitwise-equal eager step's export
            Oe = [torch.empty(w.shape, dtype=torch.float32, device=dev) for w in Ws]
            probe = B.MuonStep(0)
            Wp, Mp = [w.to(dev) for w in W0], [m.to(dev) for m in M0]
            probe.step(Wp, Gs, Mp, lrs, Oe)
            torch.cuda.synchronize()
            probe.close()
            for i in range(len(Ws)):
                assert torch.equal(Wp[i], Wg[i]) and torch.equal(Mp[i], Mg[i])
                res = oracle_for(W0[i], Gs[i].cpu(), M0[i], lrs[i])
                check_matrix(W0[i], Gs[i].cpu(), M0[i], lrs[i], Wg[i].cpu(), Mg[i].cpu(), Oe[i].cpu(), res, 2e-2,
                             f"{name}[{i}] graph")
        for a, b in zip(We, Wg):
            assert torch.equal(a.float(), b.float())
        for a, b in zip(Me, Mg):
            assert torch.equal(a, b)
    eager.close()
    graphed.close()
