"""Seeded random batches against the fp64 oracle: sizes that cross the 32-,
128- and 256-row tile boundaries at random, both orientations, padded leading
dimensions and both weight dtypes in one ragged batch."""
import numpy as np
import pytest
import torch

from muon_newton_schulz_gb300 import binding as B
from gpu_helpers import check_matrix, oracle_for

pytestmark = pytest.mark.gpu


def _batch(seed, count):
    """Host tensors of `count` random matrices and, per matrix, the padding
    of its device copies' leading dimension."""
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    Ws, Gs, Ms, lrs, pads = [], [], [], [], []
    for _ in range(count):
        m = int(rng.integers(1, 600))
        n = int(rng.integers(m, 4 * m + 64))
        rows, cols = (n, m) if rng.random() < 0.5 else (m, n)
        W = torch.randn(rows, cols, generator=g) * 0.02
        Ws.append(W.to(torch.bfloat16) if rng.random() < 0.5 else W)
        Gs.append(torch.randn(rows, cols, generator=g))
        Ms.append(torch.randn(rows, cols, generator=g) * 0.5)
        lrs.append(float(10 ** rng.uniform(-4, -2)))
        pads.append(int(rng.integers(0, 3)) * 8)
    return Ws, Gs, Ms, lrs, pads


def _to_dev(t, pad, dev):
    """Device copy whose leading dimension is the width rounded up to 8 plus
    `pad` (16-byte multiples for every dtype)."""
    ld = (t.shape[1] + 7) // 8 * 8 + pad
    full = torch.zeros(t.shape[0], ld, dtype=t.dtype, device=dev)
    full[:, :t.shape[1]] = t.to(dev)
    return full[:, :t.shape[1]]


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
@pytest.mark.parametrize("seed", [101, 202])
def test_random_ragged_batches(seed, mode):
    tol = 2e-2 if mode == B.MUON_MODE_BF16 else 1e-4
    Ws, Gs, Ms, lrs, pads = _batch(seed, 12)
    dev = torch.device("cuda", 0)
    Wd = [_to_dev(w, p, dev) for w, p in zip(Ws, pads)]
    Gd = [_to_dev(x, p, dev) for x, p in zip(Gs, pads)]
    Md = [_to_dev(x, p, dev) for x, p in zip(Ms, pads)]
    Od = [_to_dev(torch.zeros(w.shape), p, dev) for w, p in zip(Ws, pads)]
    ms = B.MuonStep(0, mode=mode)
    ms.step(Wd, Gd, Md, lrs, Od)
    torch.cuda.synchronize(dev)
    assert ms.check_status() == B.MUON_OK
    errs = []
    for i in range(len(Ws)):
        W0, G0, M0 = Ws[i], Gs[i], Ms[i]
        res = oracle_for(W0, G0, M0, lrs[i])
        errs.append(check_matrix(W0, G0, M0, lrs[i], Wd[i].cpu(), Md[i].cpu(), Od[i].cpu(), res, tol,
                                 f"seed {seed} [{i}] {tuple(W0.shape)}"))
    print(f"\nERR fuzz seed={seed} mode={mode} shapes={[tuple(w.shape) for w in Ws]} max_rel_err={max(errs):.3e}")
    ms.close()
