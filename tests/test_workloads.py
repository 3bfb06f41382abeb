"""Seeded input generators: determinism, shapes, and the spectra the
workloads ask for (log-uniform singular values, Haar singular vectors)."""
import math

import numpy as np
import torch

from muon_newton_schulz_gb300 import workloads as wl


def test_same_seed_same_inputs():
    spec = wl.MatrixSpec(16, 40, 1, "gauss", 1e-3)
    a = wl.make_matrix(spec, 7)
    b = wl.make_matrix(spec, 7)
    c = wl.make_matrix(spec, 8)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[1], c[1])


def test_dtypes_and_shapes():
    W, G, M = wl.make_matrix(wl.MatrixSpec(12, 30, 1, "gauss", w_dtype="bf16"), 1)
    assert W.dtype == torch.bfloat16 and G.dtype == torch.float32 and M.dtype == torch.float32
    assert W.shape == G.shape == M.shape == (12, 30)
    assert torch.count_nonzero(M) == 0
    W, G, M = wl.make_matrix(wl.MatrixSpec(12, 30, 1, "gauss", w_dtype="f32"), 1, steady_momentum=True)
    assert W.dtype == torch.float32 and torch.count_nonzero(M) > 0


def test_svd_spectrum_in_range():
    spec = wl.MatrixSpec(48, 20, 1, "svd", log10_lo=-5.0)
    _, G, _ = wl.make_matrix(spec, 3)
    s = np.linalg.svd(G.double().numpy(), compute_uv=False)
    assert len(s) == 20
    assert s.max() <= 1.0 + 1e-5 and s.min() >= 10 ** -5 * (1 - 1e-2)
    # Haar factors: G^T G has eigenvalues s^2 and G is built from orthonormal columns
    assert abs(np.linalg.norm(G.double().numpy()) - math.sqrt((s ** 2).sum())) < 1e-5


def test_headline_flops():
    w = wl.WORKLOADS[wl.HEADLINE]
    assert w.n_matrices == 16
    assert math.isclose(wl.workload_flops(w), 8.94e12, rel_tol=2e-3)
    assert math.isclose(wl.workload_flops(w, symmetric=False), 1.24e13, rel_tol=5e-3)


def test_workload_indices_subset():
    w = wl.WORKLOADS["ragged_h384"]
    Ws, Gs, Ms, lrs = wl.make_workload(w, indices={0, 7, 10})
    assert [tuple(g.shape) for g in Gs] == [(384, 128), (384, 384), (128, 384)]
    full = wl.make_workload(w)
    assert torch.equal(full[1][7], Gs[1])
