"""A ``torch.optim.Optimizer`` front end for the library's Muon step.

Every 2-D parameter with a gradient becomes one matrix of one ragged batch,
and one ``muon_step`` call per ``step()`` runs the momentum update, the
Newton-Schulz orthogonalisation and the weight update for all of them in the
library's kernels (EU-1T, optimizer-state paragraph: Muon on whole matrices
with one fp32 momentum state; ZAYA1/MI300X section 4.3: the update scale
0.2 * sqrt(max(rows, cols)) times the learning rate).

Parameters stay where they are: bf16 or fp32, row-major (unit column
stride), all on one CUDA device.  Each keeps an fp32 momentum buffer in the
optimizer state (``state[p]["momentum_buffer"]``).  The library reads
gradients in fp32; a gradient of another dtype (a bf16 parameter's is bf16)
or layout is first copied into an fp32 buffer kept in the state.
"""
from __future__ import annotations

import torch

from . import binding as B


class Muon(torch.optim.Optimizer):
    """Muon on 2-D parameters.

    ``lr`` may differ per parameter group.  ``beta``, ``nesterov``,
    ``dampening``, ``ns_iters``, the Newton-Schulz coefficients ``(a, b, c)``,
    ``eps`` and ``scale_coeff`` are fixed for the optimizer (the library's
    handle is configured once).  Raises ValueError for a parameter that is
    not a 2-D bf16 / fp32 CUDA tensor with unit column stride, or for
    parameters on more than one device."""

    def __init__(self, params, lr: float = 2e-4, beta: float = 0.95, nesterov: bool = False,
                 dampening: bool = False, ns_iters: int = 5, a: float = 3.4445, b: float = -4.7750,
                 c: float = 2.0315, eps: float = 1e-7, scale_coeff: float = 0.2):
        if not lr >= 0.0:
            raise ValueError(f"invalid learning rate {lr}")
        super().__init__(params, dict(lr=lr))
        devices = set()
        for group in self.param_groups:
            for p in group["params"]:
                if p.dim() != 2:
                    raise ValueError(f"Muon steps 2-D parameters only, got shape {tuple(p.shape)}")
                if p.dtype not in (torch.bfloat16, torch.float32):
                    raise ValueError(f"parameters must be bf16 or fp32, got {p.dtype}")
                if p.device.type != "cuda":
                    raise ValueError(f"parameters must be CUDA tensors, got one on {p.device}")
                if p.stride(1) != 1:
                    raise ValueError("parameters must have unit column stride (row-major)")
                devices.add(p.device.index)
        if len(devices) > 1:
            raise ValueError(f"parameters on more than one device: {sorted(devices)}")
        device = devices.pop() if devices else torch.cuda.current_device()
        self._muon = B.MuonStep(device, beta=beta, a=a, b=b, c=c, eps=eps, scale_coeff=scale_coeff,
                                ns_iters=ns_iters, nesterov=nesterov, dampening=dampening)

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        Ws, Gs, Ms, lrs = [], [], [], []
        for group in self.param_groups:
            for p in group["params"]:
                if p.grad is None:
                    continue
                state = self.state[p]
                if "momentum_buffer" not in state:
                    state["momentum_buffer"] = torch.zeros(p.shape, dtype=torch.float32, device=p.device)
                g = p.grad
                if g.dtype != torch.float32 or g.stride(1) != 1:
                    buf = state.get("grad_fp32")
                    if buf is None:
                        buf = state["grad_fp32"] = torch.empty(p.shape, dtype=torch.float32, device=p.device)
                    buf.copy_(g)
                    g = buf
                Ws.append(p)
                Gs.append(g)
                Ms.append(state["momentum_buffer"])
                lrs.append(group["lr"])
        if Ws:
            self._muon.step(Ws, Gs, Ms, lrs)
        return loss

    def check_status(self) -> int:
        """Synchronises the current stream and returns MUON_OK, or
        MUON_ERR_TIMEOUT if a kernel of an earlier step gave up a bounded
        wait (that step left W unchanged if the time-out came before its last
        kernel started)."""
        return self._muon.check_status()
