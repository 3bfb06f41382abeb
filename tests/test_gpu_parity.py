"""CUDA path against the fp64 oracle on seeded workloads small enough for
the oracle, spanning several tiles and ragged edges: tolerance 2e-2 relative
Frobenius error of O in bf16 mode and 1e-4 in the fp32 validation mode;
momentum within one fp32 ulp; weights equal to the rounded update of the
exported O."""
import pytest

from muon_newton_schulz_gb300 import binding as B
from gpu_helpers import run_and_check

pytestmark = pytest.mark.gpu

SMALL = ["single_256x512", "experts_4x256x1024", "dense_768x768", "ragged_h384", "odd_shapes"]


@pytest.mark.parametrize("name", SMALL)
def test_fp32_validation_mode(name):
    errs = run_and_check(name, mode=B.MUON_MODE_FP32_VALIDATE, tol_o=1e-4)
    assert max(errs) <= 1e-4


@pytest.mark.parametrize("name", SMALL)
def test_bf16_mode(name):
    errs = run_and_check(name, mode=B.MUON_MODE_BF16, tol_o=2e-2)
    assert max(errs) <= 2e-2


@pytest.mark.parametrize("iters", [0, 1, 2])
@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_iteration_counts(iters, mode):
    tol = 2e-2 if mode == B.MUON_MODE_BF16 else 1e-4
    run_and_check("odd_shapes", mode=mode, tol_o=tol, ns_iters=iters)


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_nesterov(mode):
    tol = 2e-2 if mode == B.MUON_MODE_BF16 else 1e-4
    run_and_check("experts_4x256x1024", mode=mode, tol_o=tol, nesterov=True, steady_momentum=True)


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_steady_state_momentum(mode):
    tol = 2e-2 if mode == B.MUON_MODE_BF16 else 1e-4
    run_and_check("ragged_h384", mode=mode, tol_o=tol, steady_momentum=True)


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_phases_split_over_launches(mode):
    """21 shape groups and 70 matrices: each Newton-Schulz phase takes two
    launches (16 + 5 groups) and the momentum pass two (64 + 6 matrices); the
    chained launches must give every matrix the oracle's result."""
    tol = 2e-2 if mode == B.MUON_MODE_BF16 else 1e-4
    runner = B.MuonStep(0, mode=mode)
    before = B.muon_launch_count(runner.h)
    errs = run_and_check("many_groups", mode=mode, tol_o=tol, runner=runner)
    launches = B.muon_launch_count(runner.h) - before
    runner.close()
    assert max(errs) <= tol
    # momentum + finalize per chunk, 3 phases x 5 iterations x 2 launches,
    # and (validation mode) a separate apply per chunk
    assert launches == 2 * 2 + 3 * 5 * 2 + (2 if mode == B.MUON_MODE_FP32_VALIDATE else 0)


@pytest.mark.parametrize("nesterov", [False, True])
@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_dampened_momentum(mode, nesterov):
    """The moving-average momentum variant (1 - beta) G, from a mid-training
    momentum state: M within one fp32 ulp of the oracle, O within tolerance."""
    tol = 2e-2 if mode == B.MUON_MODE_BF16 else 1e-4
    run_and_check("ragged_h384", mode=mode, tol_o=tol, nesterov=nesterov, dampening=True, steady_momentum=True)


@pytest.mark.parametrize("mode", [B.MUON_MODE_BF16, B.MUON_MODE_FP32_VALIDATE])
def test_extreme_aspect_ratios(mode):
    """Very long contractions and degenerate sizes: Gram X X^T with K = 100000
    (1563 k-blocks, the last one half outside the matrix), a tall 100000 x 48
    matrix (transposed in the momentum kernel and back through the W tensor
    map), one row of 300000, and a 4 x 4 matrix; all against the oracle."""
    import torch
    from muon_newton_schulz_gb300 import workloads as wl
    from gpu_helpers import check_matrix, oracle_for, run_gpu
    tol = 2e-2 if mode == B.MUON_MODE_BF16 else 1e-4
    specs = [(64, 100000, "bf16"), (100000, 48, "f32"), (1, 300000, "bf16"), (4, 4, "f32")]
    Ws, Gs, Ms, lrs = [], [], [], []
    for k, (r, c, wdt) in enumerate(specs):
        spec = wl.MatrixSpec(r, c, 1, "gauss", 1e-3, w_dtype=wdt)
        W, G, M = wl.make_matrix(spec, 91000 + k, "cpu", steady_momentum=True)
        Ws.append(W); Gs.append(G); Ms.append(M); lrs.append(2e-4)
    Wg, Mg, Og = run_gpu(Ws, Gs, Ms, lrs, mode=mode)
    for i in range(len(Ws)):
        res = oracle_for(Ws[i], Gs[i], Ms[i], lrs[i])
        check_matrix(Ws[i], Gs[i], Ms[i], lrs[i], Wg[i], Mg[i], Og[i], res, tol, f"{tuple(Ws[i].shape)}")
