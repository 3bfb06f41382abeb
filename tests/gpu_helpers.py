"""Shared helpers of the GPU tests: run the CUDA path through the C ABI on
seeded workloads and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle.muon_oracle as O
from muon_newton_schulz_gb300 import binding as B
from muon_newton_schulz_gb300 import workloads as wl

DEV = 0


def rel_frob(x, y) -> float:
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    den = np.linalg.norm(y)
    return float(np.linalg.norm(x - y) / den) if den > 0 else float(np.linalg.norm(x))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().astype(np.int32)


def f32_ulps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in fp32 units in the last place (same sign assumed)."""
    ia = a.astype(np.float32).view(np.int32).astype(np.int64)
    ib = b.astype(np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def run_gpu(Ws, Gs, Ms, lrs, mode=B.MUON_MODE_BF16, ns_iters=5, nesterov=False, export_o=True, runner=None,
            dampening=False):
    """Copies the host tensors to the GPU, runs one step and returns host
    copies (W, M, O lists).  Inputs are not modified."""
    dev = torch.device("cuda", DEV)
    Wd = [w.to(dev).contiguous() for w in Ws]
    Gd = [g.to(dev).contiguous() for g in Gs]
    Md = [m.to(dev).contiguous() for m in Ms]
    Od = [torch.full(w.shape, float("nan"), dtype=torch.float32, device=dev) for w in Ws] if export_o else None
    ms = runner or B.MuonStep(DEV, ns_iters=ns_iters, nesterov=nesterov, mode=mode, dampening=dampening)
    ms.step(Wd, Gd, Md, lrs, Od)
    torch.cuda.synchronize(dev)
    assert ms.check_status() == B.MUON_OK
    out = ([w.cpu() for w in Wd], [m.cpu() for m in Md], [o.cpu() for o in Od] if export_o else None)
    if runner is None:
        ms.close()
    return out


def oracle_for(W, G, M, lr, ns_iters=5, nesterov=False, dampening=False):
    cfg = O.OracleConfig(ns_iters=ns_iters, nesterov=nesterov, dampening=dampening)
    return O.muon_step_matrix(W.float().numpy(), G.numpy(), M.numpy(), lr, cfg, w_is_bf16=(W.dtype == torch.bfloat16))


def check_matrix(W0, G, M0, lr, Wg, Mg, Og, res, tol_o, mode_name=""):
    """Checks one matrix of a GPU step against the oracle result ``res``."""
    r, c = W0.shape
    # momentum: the fp32 fused multiply-add, within one ulp of the oracle's
    # single rounding of beta*M + G
    d = f32_ulps(Mg.numpy(), res.M)
    assert d.max() <= 1, f"{mode_name} momentum off by {d.max()} ulp"
    # orthogonalised update
    e = rel_frob(Og.numpy(), res.O)
    assert e <= tol_o, f"{mode_name} {r}x{c}: rel Frobenius error of O {e:.3e} > {tol_o}"
    # weight update from the exported O: W_gpu = round(W0 - lr_eff * O_gpu)
    # the library forms lr_eff in double from the fp32 lr and fp32 0.2, then rounds to fp32
    lr_eff = np.float32(float(np.float32(lr)) * float(np.float32(0.2)) * np.sqrt(float(max(r, c))))
    Og64 = Og.numpy().astype(np.float64)
    if W0.dtype == torch.bfloat16:
        want = O.round_to_bf16(W0.float().numpy().astype(np.float64) - float(lr_eff) * Og64)
        got = Wg.float().numpy()
        mism = got.view(np.int32) != want.view(np.int32)
        # the kernel rounds the fp32 fma result to bf16 (two roundings):
        # mismatches only at near-ties, and never more than one bf16 ulp
        assert mism.mean() <= 1e-3, f"W mismatch fraction {mism.mean():.2e}"
        if mism.any():
            dif = np.abs(bf16_bits(Wg)[mism] - bf16_bits(torch.from_numpy(want).to(torch.bfloat16))[mism])
            assert dif.max() <= 1
    else:
        want = (W0.numpy().astype(np.float64) - float(lr_eff) * Og64).astype(np.float32)
        d = f32_ulps(Wg.numpy(), want)
        assert d.max() <= 1
    return e


def run_and_check(workload_name, mode=B.MUON_MODE_BF16, tol_o=2e-2, ns_iters=5, indices=None, nesterov=False,
                  steady_momentum=False, runner=None, dampening=False):
    w = wl.WORKLOADS[workload_name]
    Ws, Gs, Ms, lrs = wl.make_workload(w, "cpu", steady_momentum=steady_momentum, indices=indices)
    Wg, Mg, Og = run_gpu(Ws, Gs, Ms, lrs, mode=mode, ns_iters=ns_iters, nesterov=nesterov, runner=runner,
                         dampening=dampening)
    errs = []
    for i in range(len(Ws)):
        res = oracle_for(Ws[i], Gs[i], Ms[i], lrs[i], ns_iters, nesterov, dampening)
        errs.append(check_matrix(Ws[i], Gs[i], Ms[i], lrs[i], Wg[i], Mg[i], Og[i], res, tol_o,
                                 f"{workload_name}[{i}]"))
    print(f"\nERR {workload_name} mode={mode} iters={ns_iters} nesterov={nesterov} dampening={dampening} "
          f"max_rel_err={max(errs):.3e}")
    return errs
