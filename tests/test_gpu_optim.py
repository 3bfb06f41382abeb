"""The torch.optim front end (muon_newton_schulz_gb300.optim.Muon) runs the
library's step on a model's 2-D parameters: two steps equal the same steps
through MuonStep bit for bit (W, momentum), with bf16 and fp32 weights and
gradients of their dtype (bf16 ones converted to fp32), two parameter groups with their own
learning rates, and a parameter without a gradient left alone."""
import pytest
import torch

from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300.optim import Muon

pytestmark = pytest.mark.gpu


def _params(dev):
    g = torch.Generator(device="cpu").manual_seed(9100)
    shapes = [(64, 160, torch.bfloat16), (160, 64, torch.float32), (96, 96, torch.bfloat16), (40, 72, torch.float32)]
    ps = []
    for r, c, dt in shapes:
        w = (torch.randn(r, c, generator=g) * 0.02).to(dt).to(dev)
        ps.append(torch.nn.Parameter(w))
    grads = [torch.randn(p.shape, generator=g) * 1e-3 for p in ps]
    return ps, grads


def test_optimizer_equals_direct_steps():
    dev = torch.device("cuda", 0)
    ps, grads = _params(dev)
    # reference: the same matrices through MuonStep
    Wr = [p.detach().clone() for p in ps]
    Mr = [torch.zeros(p.shape, dtype=torch.float32, device=dev) for p in ps]
    lrs = [2e-4, 2e-4, 5e-4, None]          # the last parameter gets no gradient
    direct = B.MuonStep(0)
    opt = Muon([{"params": ps[:2], "lr": 2e-4}, {"params": ps[2:], "lr": 5e-4}])
    for step in range(2):
        Gs = []
        for i, p in enumerate(ps):
            if lrs[i] is None:
                p.grad = None
                continue
            # a gradient has its parameter's dtype: the bf16 weights get bf16
            # gradients, which the optimizer converts to fp32
            p.grad = (grads[i] * (1.0 + step)).to(dev).to(p.dtype)
            Gs.append(p.grad.float())
        opt.step()
        idx = [i for i in range(len(ps)) if lrs[i] is not None]
        direct.step([Wr[i] for i in idx], Gs, [Mr[i] for i in idx], [lrs[i] for i in idx])
        torch.cuda.synchronize()
        assert opt.check_status() == B.MUON_OK
        for i in idx:
            assert torch.equal(ps[i].detach(), Wr[i]), (step, i)
            assert torch.equal(opt.state[ps[i]]["momentum_buffer"], Mr[i]), (step, i)
    # never stepped: unchanged, no state
    assert torch.equal(ps[3].detach(), Wr[3])
    assert ps[3] not in opt.state


def test_closure_and_empty_step():
    dev = torch.device("cuda", 0)
    ps, _ = _params(dev)
    opt = Muon(ps)
    w0 = [p.detach().clone() for p in ps]
    assert opt.step(lambda: 3.5) == 3.5      # no gradients: nothing stepped
    torch.cuda.synchronize()
    assert all(torch.equal(p.detach(), w) for p, w in zip(ps, w0))
