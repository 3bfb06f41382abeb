"""muon_step issues only kernel launches on the caller's stream (no host
synchronisation, allocation or copy), so a step can be captured in a CUDA
graph and replayed: replays give bitwise the results of eager steps."""
import pytest
import torch

from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl

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
    for _ in range(3):
        eager.step(We, Gs, Me, lrs)
        graph.replay()
        torch.cuda.synchronize()
        for a, b in zip(We, Wg):
            assert torch.equal(a.float(), b.float())
        for a, b in zip(Me, Mg):
            assert torch.equal(a, b)
    eager.close()
    graphed.close()
