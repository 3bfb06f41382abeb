"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formulas: each compares it with an
independent fact -- the SVD form of a matrix polynomial, the polar factor
from scipy, exact rational arithmetic, explicit triple loops, equivariances
and torch's bf16 cast.  The last group plants plausible mistakes in a copy of
the oracle and checks that the pins catch each of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle.muon_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")
A, B, C = O.NS_A, O.NS_B, O.NS_C


def _rng(seed):
    return np.random.default_rng(seed)


def _svd_closed_form(X, a, b, c, iters, eps):
    """U diag(p^iters(sigma / (||X||_F + eps))) V^T, with the scalar map
    p(s) = a s + b s^3 + c s^5 applied to each singular value."""
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    s = s / (np.linalg.norm(X) + eps)
    for _ in range(iters):
        s = a * s + b * s ** 3 + c * s ** 5
    return (U * s) @ Vt


def _oracle_O(G, cfg=O.OracleConfig()):
    r, c = G.shape
    res = O.muon_step_matrix(np.zeros((r, c), np.float32), G.astype(np.float32),
                             np.zeros((r, c), np.float32), 0.0, cfg)
    return res.O


def _rel(x, y):
    return np.linalg.norm(x - y) / max(np.linalg.norm(y), 1e-300)


# --- closed form through the SVD -------------------------------------------------

@pytest.mark.parametrize("shape", [(8, 12), (16, 16), (24, 10), (1, 7), (9, 1)])
def test_svd_polynomial_closed_form(shape):
    G = _rng(sum(shape)).standard_normal(shape).astype(np.float32)
    got = _oracle_O(G)
    want = _svd_closed_form(G.astype(np.float64), A, B, C, 5, 1e-7)
    assert _rel(got, want) < 1e-10


@pytest.mark.parametrize("iters", [0, 1, 2, 7])
def test_svd_closed_form_any_iteration_count(iters):
    G = _rng(7).standard_normal((6, 11)).astype(np.float32)
    got = _oracle_O(G, O.OracleConfig(ns_iters=iters))
    want = _svd_closed_form(G.astype(np.float64), A, B, C, iters, 1e-7)
    assert _rel(got, want) < 1e-10


def test_svd_closed_form_ill_conditioned():
    r = _rng(3)
    U, _ = np.linalg.qr(r.standard_normal((12, 12)))
    V, _ = np.linalg.qr(r.standard_normal((20, 12)))
    s = 10.0 ** r.uniform(-5, 0, 12)
    G = ((U * s) @ V.T).astype(np.float32)
    got = _oracle_O(G)
    want = _svd_closed_form(G.astype(np.float64), A, B, C, 5, 1e-7)
    assert _rel(got, want) < 1e-10


# --- textbook special case: cubic Newton-Schulz converges to the polar factor ----

@pytest.mark.parametrize("shape", [(6, 10), (10, 6), (8, 8)])
def test_polar_factor_limit(shape):
    G = _rng(11 + shape[0]).standard_normal(shape)
    X, transposed = O.orient(G)
    X = O.frobenius_normalise(X, 0.0)
    for _ in range(100):
        Xn = O.ns_iteration(X, 1.5, -0.5, 0.0)
        done = np.linalg.norm(Xn - X) < 1e-13
        X = Xn
        if done:
            break
    Q = X.T if transposed else X
    upol, _ = scipy.linalg.polar(G, side="right")
    assert np.abs(Q - upol).max() < 1e-11
    Us, _, Vt = np.linalg.svd(G, full_matrices=False)
    assert np.abs(Q - Us @ Vt).max() < 1e-11


# --- exact symmetry -------------------------------------------------------------

def test_gram_products_exactly_symmetric():
    X = _rng(5).standard_normal((33, 71))
    Am = O.sym_upper(X)
    assert np.array_equal(Am, Am.T)
    A2 = O.sym_upper(Am)
    assert np.array_equal(A2, A2.T)
    # the kept triangle is the upper one of the plain product
    full = X @ X.T
    iu = np.triu_indices(33)
    assert np.array_equal(Am[iu], full[iu])


# --- invariants ------------------------------------------------------------------

def test_scale_invariance():
    G = _rng(21).standard_normal((10, 14))
    cfg = O.OracleConfig(eps=0.0)
    o1 = _oracle_O(G.astype(np.float32), cfg)
    o2 = _oracle_O((G * 8.0).astype(np.float32), cfg)  # power of two: exact in fp32
    assert _rel(o2, o1) < 1e-12


def test_transpose_equivariance_rectangular():
    # both orientations reduce to the same wide X, so only BLAS summation
    # order (strided vs contiguous operands) can differ
    G = _rng(22).standard_normal((9, 15)).astype(np.float32)
    o = _oracle_O(G)
    ot = _oracle_O(np.ascontiguousarray(G.T))
    assert ot.shape == (15, 9)
    assert _rel(ot, o.T) < 1e-13


def test_transpose_equivariance_square():
    G = _rng(23).standard_normal((12, 12)).astype(np.float32)
    o = _oracle_O(G)
    ot = _oracle_O(np.ascontiguousarray(G.T))
    assert _rel(ot, o.T) < 1e-10


def test_orthogonal_equivariance():
    r = _rng(24)
    G = r.standard_normal((7, 13))
    Q, _ = np.linalg.qr(r.standard_normal((7, 7)))
    R, _ = np.linalg.qr(r.standard_normal((13, 13)))
    cfg = O.OracleConfig(eps=0.0)
    X = O.frobenius_normalise(G, 0.0)
    lhs = O.newton_schulz(O.frobenius_normalise(Q @ G @ R, 0.0), A, B, C, 5)
    rhs = Q @ O.newton_schulz(X, A, B, C, 5) @ R
    assert _rel(lhs, rhs) < 1e-10
    assert cfg.eps == 0.0


def test_rank_preserved():
    # small-integer factors: the rank-3 product is exact in fp32
    r = _rng(25)
    G = r.integers(-4, 5, (10, 3)).astype(np.float64) @ r.integers(-4, 5, (3, 16)).astype(np.float64)
    assert np.linalg.matrix_rank(G) == 3
    o = _oracle_O(G.astype(np.float32))
    s = np.linalg.svd(o, compute_uv=False)
    assert np.all(s[:3] > 1e-3)
    assert np.all(s[3:] < 1e-10)


def test_zero_gradient_gives_zero_update():
    W = _rng(26).standard_normal((5, 9)).astype(np.float32)
    Z = np.zeros((5, 9), np.float32)
    res = O.muon_step_matrix(W, Z, Z, 1e-2)
    assert np.all(res.O == 0.0)
    assert np.array_equal(res.W, W)
    assert np.all(res.M == 0.0)


def test_momentum_closed_form():
    r = _rng(27)
    beta = float(np.float32(0.95))
    Gs = [r.standard_normal((4, 6)).astype(np.float32) for _ in range(6)]
    M = np.zeros((4, 6), np.float32)
    for G in Gs:
        M = O.momentum(M, G, beta)
    t = len(Gs)
    want = sum(beta ** (t - 1 - k) * Gs[k].astype(np.float64) for k in range(t))
    assert np.abs(M - want).max() <= 8 * np.finfo(np.float32).eps * np.abs(want).max()


def test_momentum_is_a_single_rounding():
    """beta*M + G is exact in fp64 for these inputs, so the oracle's fp32 value
    is the correctly rounded one: compare with exact rationals."""
    r = _rng(28)
    beta = float(np.float32(0.95))
    M = r.standard_normal(200).astype(np.float32)
    G = r.standard_normal(200).astype(np.float32)
    got = O.momentum(M, G, beta)
    for i in range(200):
        exact = Fraction(beta) * Fraction(float(M[i])) + Fraction(float(G[i]))
        cand = np.float32(float(exact))
        # the nearest fp32 to the exact value
        lo, hi = np.nextafter(cand, np.float32(-np.inf)), np.nextafter(cand, np.float32(np.inf))
        best = min((cand, lo, hi), key=lambda v: abs(Fraction(float(v)) - exact))
        assert got[i] == best


# --- brute force -----------------------------------------------------------------

def _loops_matmul(P, Q):
    n, k = P.shape
    k2, m = Q.shape
    assert k == k2
    out = np.zeros((n, m))
    for i in range(n):
        for j in range(m):
            acc = 0.0
            for t in range(k):
                acc += P[i, t] * Q[t, j]
            out[i, j] = acc
    return out


def test_bruteforce_iteration():
    X = _rng(31).standard_normal((4, 6))
    # Gram product by loops, upper triangle mirrored
    Am = _loops_matmul(X, X.T)
    for i in range(4):
        for j in range(i):
            Am[i, j] = Am[j, i]
    A2 = _loops_matmul(Am, Am)
    want = A * X + B * _loops_matmul(Am, X) + C * _loops_matmul(A2, X)
    got = O.ns_iteration(X, A, B, C)
    assert np.abs(got - want).max() < 1e-13
    assert np.abs(O.sym_upper(X) - Am).max() < 1e-13


def test_folded_association_matches():
    X = O.frobenius_normalise(_rng(32).standard_normal((20, 37)), 0.0)
    assert _rel(O.ns_iteration_folded(X, A, B, C), O.ns_iteration(X, A, B, C)) < 1e-12


# --- exact scalar values ---------------------------------------------------------

def test_scalar_polynomial_exact():
    a, b, c = (Fraction(str(v)) for v in (A, B, C))
    p = lambda s: a * s + b * s ** 3 + c * s ** 5
    assert p(Fraction(1)) == Fraction("0.701")
    assert a + 3 * b + 5 * c == Fraction("-0.723")  # p'(1)
    # a single row vector has one singular value, 1 after normalisation
    v = np.array([[3.0, 4.0, 0.0, 12.0]], dtype=np.float32)  # norm 13
    s = Fraction(1)
    for _ in range(5):
        s = p(s)
    res = _oracle_O(v, O.OracleConfig(eps=0.0))
    assert np.abs(res - float(s) * v.astype(np.float64) / 13.0).max() < 1e-14


def test_update_scale_values():
    assert O.update_scale(100, 25) == pytest.approx(2.0, abs=1e-15)
    assert O.update_scale(64, 4096) == pytest.approx(12.8, abs=1e-14)
    assert O.update_scale(4096, 64) == O.update_scale(64, 4096)


def test_weight_update_formula():
    """With cubic coefficients run to convergence O is the polar factor, so
    the update is exactly lr * 0.2 * sqrt(max) * U V^T."""
    r = _rng(33)
    G = r.standard_normal((6, 16)).astype(np.float32)
    W = r.standard_normal((6, 16)).astype(np.float32)
    cfg = O.OracleConfig(a=1.5, b=-0.5, c=0.0, ns_iters=60, eps=0.0)
    res = O.muon_step_matrix(W, G, np.zeros_like(G), 0.01, cfg)
    Us, _, Vt = np.linalg.svd(G.astype(np.float64), full_matrices=False)
    want = (W.astype(np.float64) - 0.01 * 0.2 * 4.0 * (Us @ Vt)).astype(np.float32)
    assert np.abs(res.W - want).max() < 1e-6


def test_page_constants_fixture():
    g = json.load(open(GOLDEN, encoding="utf-8"))
    cfg = O.OracleConfig()
    assert cfg.ns_iters == g["ns_iters_per_step"]["value"]
    assert cfg.scale_coeff == g["lr_scale_coeff"]["value"]
    from muon_newton_schulz_gb300 import workloads as wl
    assert wl.WORKLOADS["experts_16x2048x8192"].specs[0].rows == g["expert_ffn_shape"]["value"][0]
    assert wl.WORKLOADS["experts_16x2048x8192"].specs[0].cols == g["expert_ffn_shape"]["value"][1]
    assert wl.WORKLOADS["experts_16x2048x8192"].specs[0].count == g["experts_per_layer_zaya1"]["value"]
    assert wl.WORKLOADS["experts_128x2048x8192"].specs[0].count == g["experts_torchtitan"]["value"]
    assert wl.WORKLOADS["dense_7680x7680"].specs[0].rows == g["attention_qkv_shape"]["value"][0]
    assert wl.WORKLOADS["ragged_h6144"].specs[1].rows == g["hidden_1t_moe"]["value"]
    assert wl.WORKLOADS["experts_16x2048x8192"].lr == g["lr"]["value"]


# --- bf16 rounding against torch's cast --------------------------------------------

def test_round_to_bf16_matches_torch_cast():
    r = _rng(41)
    x = np.concatenate([
        r.standard_normal(20000).astype(np.float32),
        (r.standard_normal(2000) * 1e-39).astype(np.float32),     # fp32 subnormals
        (r.standard_normal(2000) * 1e38).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38,
                  1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 2.0 ** -126, 2.0 ** -133,
                  1.5 * 2.0 ** -133, 2.5 * 2.0 ** -133], np.float32),
    ])
    # ties: bf16 values with the next bit set
    ties = (torch.from_numpy(r.standard_normal(2000).astype(np.float32)).to(torch.bfloat16).float().numpy()
            .view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties])
    got = O.round_to_bf16(x.astype(np.float64))
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_round_to_bf16_from_fp64_is_direct():
    # 1 + 2^-8 + 2^-30: fp32 would round it to 1 + 2^-8 (a tie, then to 1);
    # directly from fp64 it is above the tie and goes up.
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30])
    assert O.round_to_bf16(x)[0] == np.float32(1.0 + 2.0 ** -7)


# --- planted mistakes are caught ---------------------------------------------------

def _mutant_iterations():
    def drop_c(X, a, b, c):
        Am = O.sym_upper(X)
        return a * X + b * (Am @ X)

    def sign_b(X, a, b, c):
        Am = O.sym_upper(X)
        A2 = O.sym_upper(Am)
        return a * X - b * (Am @ X) + c * (A2 @ X)

    def wrong_gram(X, a, b, c):  # X^T X used where X X^T is meant
        Am = X.T @ X
        A2 = Am @ Am
        return a * X + b * (X @ Am) + c * (X @ A2) * 1.0001

    def lower_triangle_wrong(X, a, b, c):  # mirrors the wrong triangle of A2
        Am = O.sym_upper(X)
        full = Am @ Am
        A2 = np.triu(full) + np.triu(full, 1)  # not mirrored: upper only
        return a * X + b * (Am @ X) + c * (A2 @ X)

    return [drop_c, sign_b, wrong_gram, lower_triangle_wrong]


@pytest.mark.parametrize("mutant", _mutant_iterations(), ids=lambda f: f.__name__)
def test_planted_mistakes_fail_the_svd_pin(mutant, monkeypatch):
    monkeypatch.setattr(O, "ns_iteration", mutant)
    G = _rng(51).standard_normal((8, 12)).astype(np.float32)
    got = _oracle_O(G)
    want = _svd_closed_form(G.astype(np.float64), A, B, C, 5, 1e-7)
    assert not (_rel(got, want) <= 1e-6)


def test_planted_missing_normalisation_fails(monkeypatch):
    monkeypatch.setattr(O, "frobenius_normalise", lambda X, eps: X)
    G = (_rng(52).standard_normal((8, 12)) * 0.05).astype(np.float32)
    got = _oracle_O(G)
    want = _svd_closed_form(G.astype(np.float64), A, B, C, 5, 1e-7)
    assert not (_rel(got, want) <= 1e-6)


def test_planted_missing_transpose_back_fails(monkeypatch):
    def orient_no_T(M):
        rows, cols = M.shape
        return (M.T.astype(np.float64), False) if rows > cols else (M.astype(np.float64), False)
    monkeypatch.setattr(O, "orient", orient_no_T)
    G = _rng(53).standard_normal((12, 8)).astype(np.float32)
    r, c = G.shape
    with pytest.raises(Exception):
        res = O.muon_step_matrix(np.zeros((r, c), np.float32), G, np.zeros((r, c), np.float32), 0.1)
        assert res.W.shape == (r, c) and res.O.shape == (r, c)


def test_nesterov_from_zero_momentum_is_a_rescaling():
    """With M = 0 the Nesterov input is (1 + beta) G, and the normalisation
    removes any positive scale (eps = 0 makes it exact)."""
    G = _rng(61).standard_normal((7, 12)).astype(np.float32)
    Z = np.zeros_like(G)
    plain = O.muon_step_matrix(Z, G, Z, 0.0, O.OracleConfig(eps=0.0))
    nest = O.muon_step_matrix(Z, G, Z, 0.0, O.OracleConfig(eps=0.0, nesterov=True))
    assert _rel(nest.O, plain.O) < 1e-12
    # with a non-zero momentum the two differ
    M = _rng(62).standard_normal((7, 12)).astype(np.float32)
    a = O.muon_step_matrix(Z, G, M, 0.0, O.OracleConfig())
    b = O.muon_step_matrix(Z, G, M, 0.0, O.OracleConfig(nesterov=True))
    assert _rel(a.O, b.O) > 1e-3
    assert np.array_equal(a.M, b.M)


def test_dampened_momentum_closed_form_and_fixed_point():
    """With dampening the momentum is the moving average
    (1 - beta) * sum_k beta^(t-1-k) G_k; a constant gradient G gives
    (1 - beta^t) G, which tends to G (reading R17)."""
    r = _rng(63)
    beta = float(np.float32(0.95))
    Gs = [r.standard_normal((4, 6)).astype(np.float32) for _ in range(6)]
    M = np.zeros((4, 6), np.float32)
    for G in Gs:
        M = O.momentum(M, G, beta, dampening=True)
    t = len(Gs)
    want = (1.0 - beta) * sum(beta ** (t - 1 - k) * Gs[k].astype(np.float64) for k in range(t))
    assert np.abs(M - want).max() <= 8 * np.finfo(np.float32).eps * np.abs(want).max()
    G = r.standard_normal((3, 5)).astype(np.float32)
    M = np.zeros_like(G)
    for _ in range(40):
        M = O.momentum(M, G, beta, dampening=True)
    want = (1.0 - beta ** 40) * G.astype(np.float64)
    assert np.abs(M - want).max() <= 64 * np.finfo(np.float32).eps * np.abs(G).max()


def test_dampened_momentum_is_a_single_rounding():
    """beta*M + (1 - beta)*G is exact in fp64 for fp32 inputs (1 - beta has 20
    significant bits), so the oracle's fp32 value is the nearest one."""
    r = _rng(64)
    beta = float(np.float32(0.95))
    M = r.standard_normal(200).astype(np.float32)
    G = r.standard_normal(200).astype(np.float32)
    got = O.momentum(M, G, beta, dampening=True)
    d = Fraction(1) - Fraction(beta)
    for i in range(200):
        exact = Fraction(beta) * Fraction(float(M[i])) + d * Fraction(float(G[i]))
        cand = np.float32(float(exact))
        lo, hi = np.nextafter(cand, np.float32(-np.inf)), np.nextafter(cand, np.float32(np.inf))
        best = min((cand, lo, hi), key=lambda v: abs(Fraction(float(v)) - exact))
        assert got[i] == best


def test_dampened_nesterov_from_zero_momentum_is_a_rescaling():
    """Dampening and Nesterov together from a zero momentum: the NS input is a
    positive multiple of G up to the fp32 rounding of the stored momentum, so
    the update equals the plain one (eps = 0) to about fp32 precision."""
    G = _rng(65).standard_normal((6, 10)).astype(np.float32)
    Z = np.zeros_like(G)
    plain = O.muon_step_matrix(Z, G, Z, 0.0, O.OracleConfig(eps=0.0))
    both = O.muon_step_matrix(Z, G, Z, 0.0, O.OracleConfig(eps=0.0, nesterov=True, dampening=True))
    assert _rel(both.O, plain.O) < 1e-6


# --- the Nesterov input, pinned by a two-step case with a closed-form answer --------
#
# G1 has one non-zero row u (row 0) and G2 one non-zero row v (row 1), with u and
# v orthogonal unit vectors whose entries are +-1/2, so every stored fp32 value
# below is exact.  From M0 = 0, two steps give M2 = beta*G1 + G2 (plain form) and
# the Nesterov input G2 + beta*M2 = beta^2 G1 + (1 + beta) G2: its rows are
# orthogonal, so its singular values are beta^2 and 1 + beta, with u and v as
# right singular vectors.  Newton-Schulz maps each normalised singular value
# s -> p(s) = a s + b s^3 + c s^5, so the update is
#     O = [p^5(beta^2 / F) u ; p^5((1 + beta) / F) v],   F = sqrt(beta^4 + (1 + beta)^2),
# evaluated here in 50-digit decimal arithmetic, independently of numpy.

U_ROW = np.array([0.5, 0.5, 0.5, 0.5])
V_ROW = np.array([0.5, -0.5, 0.5, -0.5])


def _two_step_O(cfg):
    G1 = np.zeros((2, 4), np.float32)
    G1[0] = U_ROW
    G2 = np.zeros((2, 4), np.float32)
    G2[1] = V_ROW
    Z = np.zeros((2, 4), np.float32)
    first = O.muon_step_matrix(Z, G1, Z, 0.0, cfg)
    second = O.muon_step_matrix(Z, G2, first.M, 0.0, cfg)
    return second.O


def _decimal_update(row_norms):
    """[p^5(n0 / F) u ; p^5(n1 / F) v] for the singular values n0, n1 given as
    Decimals (F their 2-norm), as float64."""
    import decimal
    with decimal.localcontext() as ctx:
        ctx.prec = 50
        D = decimal.Decimal
        a, b, c = D(str(A)), D(str(B)), D(str(C))
        n0, n1 = row_norms
        F = (n0 * n0 + n1 * n1).sqrt()
        out = []
        for n in (n0, n1):
            s = n / F
            for _ in range(5):
                s = a * s + b * s ** 3 + c * s ** 5
            out.append(float(s))
    return np.stack([out[0] * U_ROW, out[1] * V_ROW])


def _beta_decimal():
    import decimal
    return decimal.Decimal(float(np.float32(0.95)))


def test_nesterov_input_two_step_closed_form():
    import decimal
    beta = _beta_decimal()
    want = _decimal_update((beta * beta, 1 + beta))
    got = _two_step_O(O.OracleConfig(eps=0.0, nesterov=True))
    assert np.abs(got - want).max() < 1e-12
    # the plain step sees M2 itself, with singular values beta and 1
    plain = _two_step_O(O.OracleConfig(eps=0.0))
    assert np.abs(plain - _decimal_update((beta, decimal.Decimal(1)))).max() < 1e-12
    assert np.abs(got - plain).max() > 1e-3


def test_dampened_nesterov_input_two_step_closed_form():
    """With dampening, M1 = (1 - beta) G1 and M2 = beta M1 + (1 - beta) G2,
    stored in fp32: row 0 of M2 is fl32(beta (1 - beta)) u (beta (1 - beta)
    has 44 significant bits, so the stored state is rounded once), row 1 is
    (1 - beta) v.  The Nesterov input (1 - beta) G2 + beta M2 then has
    singular values beta fl32(beta (1 - beta)) and (1 - beta)(1 + beta)."""
    import decimal
    beta = _beta_decimal()
    d = 1 - beta                                   # exact in fp32 (Sterbenz)
    stored = decimal.Decimal(float(np.float32(float(beta * d))))   # fp32 storage of the momentum
    want = _decimal_update((beta * stored, d * (1 + beta)))
    got = _two_step_O(O.OracleConfig(eps=0.0, nesterov=True, dampening=True))
    assert np.abs(got - want).max() < 1e-12


def _nesterov_mutants():
    def swapped(M_new, G, beta, dampening=False):     # M_new + beta*G instead of G + beta*M_new
        g = G.astype(np.float64)
        if dampening:
            g = (1.0 - float(beta)) * g
        return M_new.astype(np.float64) + float(beta) * g

    def ignored(M_new, G, beta, dampening=False):     # no look-ahead at all
        return M_new.astype(np.float64)

    def undampened_gradient(M_new, G, beta, dampening=False):   # (1 - beta) dropped from G
        return G.astype(np.float64) + float(beta) * M_new.astype(np.float64)

    return [swapped, ignored, undampened_gradient]


@pytest.mark.parametrize("mutant", _nesterov_mutants(), ids=lambda f: f.__name__)
@pytest.mark.parametrize("dampening", [False, True])
def test_planted_nesterov_mistakes_fail_the_two_step_pin(mutant, dampening, monkeypatch):
    import decimal
    beta = _beta_decimal()
    if dampening:
        d = 1 - beta
        stored = decimal.Decimal(float(np.float32(float(beta * d))))
        want = _decimal_update((beta * stored, d * (1 + beta)))
    else:
        if mutant.__name__ == "undampened_gradient":
            pytest.skip("identical to the correct form without dampening")
        want = _decimal_update((beta * beta, 1 + beta))
    monkeypatch.setattr(O, "nesterov_input", mutant)
    got = _two_step_O(O.OracleConfig(eps=0.0, nesterov=True, dampening=dampening))
    assert not (np.abs(got - want).max() < 1e-6)
