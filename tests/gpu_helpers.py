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


def bf16_ordered(t: torch.Tensor) -> np.ndarray:
    """bf16 bit patterns mapped to integers in the order of the values they
    hold (+0 and -0 both to 0), so adjacent bf16 numbers differ by one, also
    across zero."""
    b = bf16_bits(t)
    mag = b & 0x7FFF
    return np.where(b < 0, -mag, mag)


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
            dif = np.abs(bf16_ordered(Wg)[mism] - bf16_ordered(torch.from_numpy(want).to(torch.bfloat16))[mism])
            assert dif.max() <= 1
    else:
        want = (W0.numpy().astype(np.float64) - float(lr_eff) * Og64).astype(np.float32)
        d = f32_ulps(Wg.numpy(), want)
        assert d.max() <= 1
    check_w_against_oracle(W0, Wg, Og64, res, lr_eff, mode_name)
    return e


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits; 2^-133 below the
    normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check_w_against_oracle(W0, Wg, Og64, res, lr_eff, what=""):
    """The GPU's W against the oracle's own rounded update res.W.  Both round
    an update of the same W0, and the unrounded values differ by at most
    `reach` = lr_eff * |O_gpu - O_oracle| (O agrees to the mode's tolerance)
    plus the fp32 arithmetic of the kernel, so the rounded values differ by at
    most reach plus half a unit in the last place of each.  Where reach is
    below half an ulp (the usual case) they are equal or neighbours."""
    w0 = W0.float().numpy().astype(np.float64)
    got = Wg.float().numpy().astype(np.float64)
    want = res.W.astype(np.float64)
    o_or = np.asarray(res.O, np.float64)
    x = w0 - float(lr_eff) * o_or                     # the oracle's update before rounding
    reach = (float(lr_eff) * np.abs(Og64 - o_or)       # what the O difference moves
             + 1e-6 * float(lr_eff) * np.abs(o_or)     # lr and scale formed in fp32 vs fp64
             + 4 * 2.0 ** -24 * np.abs(x))             # the kernel's fp32 fma before the final rounding
    if W0.dtype == torch.bfloat16:
        half = 0.5 * (bf16_ulp(got) + bf16_ulp(want))
    else:
        half = 2.0 ** -24 * (np.abs(got) + np.abs(want))
    err = np.abs(got - want)
    bad = err > reach + half
    assert not bad.any(), (f"{what} W off the oracle's by {err[bad].max():.3e} where the O difference allows "
                           f"{(reach + half)[bad][np.argmax(err[bad])]:.3e}")


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
