"""Plain fp64 CPU oracle of one Muon optimizer step on whole matrices.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, constant table or helper with the CUDA library; the two meet only in
the seeded input generators, which hold none of the method's arithmetic.

What it computes, step by step, for each matrix independently (numpy,
float64, one library matmul per product, no blocking or fusion):

1. Momentum.  One fp32 momentum state per parameter ("Training a 1T-Params
   MoE on EU public infrastructure", tanhow.com, the paragraph on optimizer
   state): ``M <- beta*M + G``, stored back as fp32.
2. Orientation.  ``X = M`` if rows <= cols, else ``X = M^T``, so that the Gram
   matrix ``A = X X^T`` is the smaller one (reading R5 below).
3. Frobenius normalisation ``X <- X / (||X||_F + eps)`` (reading R4).
4. Newton-Schulz, repeated ``iters`` times (5 per step: "ZAYA1 MoE training
   on MI300X", hotelren.com/news/3048137, section 4.3 训练配方细节), each
   iteration as written in "AMD GPU深度学习优化与ZAYA1大模型实践",
   jsqmd.com/news/1098463, section 4.2 内存高效Muon优化器:
   ``A = sym(X X^T)``, ``A2 = sym(A A)`` (the symmetric kernel reused),
   ``X <- a X + b A X + c A2 X``.  ``sym`` keeps the upper triangle and
   mirrors it, which is what "compute only the upper triangle" yields.
5. Orientation back: ``O = X`` or ``X^T``.
6. Update ``W <- W - lr * 0.2 * sqrt(max(rows, cols)) * O`` (hotelren.com,
   section 4.3: learning-rate scale 0.2 x sqrt(max(a, b)), a and b read as the
   matrix dimensions), in fp64, then rounded to the weight dtype with
   round-to-nearest-even.

Readings where the pages are silent (each also listed in the design notes):
  R1 coefficients (a, b, c) = (3.4445, -4.7750, 2.0315), the same every
     iteration; R2 momentum ``beta*M + G`` without dampening, beta = 0.95;
  R3 no Nesterov by default; with ``nesterov`` the NS input is
     ``G + beta*M`` (new M), the usual Nesterov form; R4 eps = 1e-7 added to the norm; R5 transpose iff
  rows > cols; R6 no weight decay; R7 bf16 weights rounded RN-even;
  R17 (a variant, off by default) ``dampening``: ``M <- beta*M + (1-beta)*G``
     and the Nesterov input ``(1-beta)*G + beta*M``.

Pins (tests/test_oracle_pins.py): the singular-value polynomial closed form
via SVD, convergence to the polar factor with (1.5, -0.5, 0) against
scipy.linalg.polar, exact symmetry, scale / transpose / orthogonal
equivariance, rank preservation, the momentum closed form, brute-force
triple-loop products, exact rational values of the scalar polynomial,
torch's fp32->bf16 cast for ``round_to_bf16``, and for ``nesterov_input`` a
two-step case with orthogonal gradient rows whose update has a closed form
(singular values beta^2 and 1 + beta), evaluated in 50-digit decimal
arithmetic.  Every function here has a pin.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

# Reading R1: the pages give no coefficients; these are the quintic ones
# commonly used for Muon, constant across iterations.
NS_A, NS_B, NS_C = 3.4445, -4.7750, 2.0315


@dataclass(frozen=True)
class OracleConfig:
    """Scalars of one step.  ``beta`` is passed exactly as the GPU side gets
    it (the fp32 value of 0.95) so that the momentum check can be bit-level."""

    beta: float = float(np.float32(0.95))
    a: float = NS_A
    b: float = NS_B
    c: float = NS_C
    eps: float = 1e-7
    scale_coeff: float = 0.2
    ns_iters: int = 5
    nesterov: bool = False
    dampening: bool = False


def momentum(M: np.ndarray, G: np.ndarray, beta: float, dampening: bool = False) -> np.ndarray:
    """Step 1: ``beta*M + G`` evaluated in fp64 from the fp32 inputs and
    rounded once to fp32.  beta*M is exact in fp64 (24+24 bit product), so this
    equals the correctly rounded fused multiply-add except in double-rounding
    corner cases.  With ``dampening`` (reading R17) the gradient enters as
    ``(1 - beta)*G``, the moving-average form; 1 - beta is exact for the fp32
    beta and its product with G is exact in fp64 too."""
    g = G.astype(np.float64)
    if dampening:
        g = (1.0 - float(beta)) * g
    out = float(beta) * M.astype(np.float64) + g
    return out.astype(np.float32)


def nesterov_input(M_new: np.ndarray, G: np.ndarray, beta: float, dampening: bool = False) -> np.ndarray:
    """Step 1b, only with ``nesterov`` (reading R3): the Newton-Schulz input
    looks one momentum step ahead, ``G + beta*M_new`` with the momentum just
    updated in step 1, evaluated in fp64 from the stored fp32 values.  With
    ``dampening`` (reading R17) the gradient term is ``(1 - beta)*G`` as in
    the momentum itself."""
    g = G.astype(np.float64)
    if dampening:
        g = (1.0 - float(beta)) * g
    return g + float(beta) * M_new.astype(np.float64)


def orient(M: np.ndarray) -> tuple[np.ndarray, bool]:
    """Step 2: wide orientation.  Returns (X, transposed)."""
    rows, cols = M.shape
    if rows > cols:
        return M.T.astype(np.float64), True
    return M.astype(np.float64), False


def frobenius_normalise(X: np.ndarray, eps: float) -> np.ndarray:
    """Step 3: ``X / (||X||_F + eps)``."""
    nrm = math.sqrt(float(np.sum(X * X)))
    return X / (nrm + eps)


def sym_upper(P: np.ndarray) -> np.ndarray:
    """``P P^T`` of which only the upper triangle is kept and then mirrored,
    so the result is exactly symmetric (the page's ``symmetric_mm``)."""
    full = P @ P.T
    upper = np.triu(full)
    return upper + np.triu(full, 1).T


def ns_iteration(X: np.ndarray, a: float, b: float, c: float) -> np.ndarray:
    """One Newton-Schulz iteration in the order the page writes it:
    A = sym(X X^T); A2 = sym(A A^T) = A^2 because A is symmetric;
    X <- a X + b (A X) + c (A2 X)."""
    A = sym_upper(X)
    A2 = sym_upper(A)
    return a * X + b * (A @ X) + c * (A2 @ X)


def ns_iteration_folded(X: np.ndarray, a: float, b: float, c: float) -> np.ndarray:
    """The same iteration associated as ``(b A + c A2) X + a X``; equal to
    ``ns_iteration`` in exact arithmetic (a pin compares the two)."""
    A = sym_upper(X)
    A2 = sym_upper(A)
    B = b * A + c * A2
    return B @ X + a * X


def newton_schulz(X: np.ndarray, a: float, b: float, c: float, iters: int) -> np.ndarray:
    """Step 4: ``iters`` iterations with the same coefficients."""
    for _ in range(iters):
        X = ns_iteration(X, a, b, c)
    return X


def update_scale(rows: int, cols: int, coeff: float = 0.2) -> float:
    """``coeff * sqrt(max(rows, cols))`` (hotelren.com, section 4.3)."""
    return coeff * math.sqrt(max(rows, cols))


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 (8 significant bits, ties to
    even, fp32 exponent range, overflow to inf), returned as float32 holding
    the bf16 value.  Written from the format's definition, rounding directly
    from fp64 (no intermediate fp32 rounding)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    out[~finite] = x[~finite]
    xf = x[finite]
    mant, expo = np.frexp(xf)  # xf = mant * 2**expo, 0.5 <= |mant| < 1
    # bf16 normal numbers: exponent of the leading bit >= -126, i.e. expo >= -125.
    # Below that the spacing is fixed at 2**-133 (subnormals).
    lsb_expo = np.maximum(expo - 8, -133)
    q = np.ldexp(xf, -lsb_expo)
    q = np.rint(q)  # numpy rint is round-half-to-even
    y = np.ldexp(q, lsb_expo)
    max_bf16 = float.fromhex("0x1.fep127")
    y = np.where(np.abs(y) > max_bf16, np.copysign(np.inf, y), y)
    out[finite] = y
    return out.astype(np.float32)


@dataclass
class OracleStepResult:
    W: np.ndarray           # updated weights, dtype of the input W (float32 holding bf16 values for bf16)
    M: np.ndarray           # updated momentum, float32
    O: np.ndarray           # orthogonalised update, fp64, rows x cols
    X0: np.ndarray          # normalised NS input, fp64, wide orientation
    scale: float            # 0.2 * sqrt(max(rows, cols))


def muon_step_matrix(W: np.ndarray, G: np.ndarray, M: np.ndarray, lr: float,
                     cfg: OracleConfig = OracleConfig(), w_is_bf16: bool = False) -> OracleStepResult:
    """Steps 1-6 for one matrix.  ``W`` is float32 (holding bf16 values when
    ``w_is_bf16``), ``G`` and ``M`` float32, all rows x cols."""
    M_new = momentum(M, G, cfg.beta, cfg.dampening)
    src = nesterov_input(M_new, G, cfg.beta, cfg.dampening) if cfg.nesterov else M_new
    X, transposed = orient(src)
    X0 = frobenius_normalise(X, cfg.eps)
    Xk = newton_schulz(X0, cfg.a, cfg.b, cfg.c, cfg.ns_iters)
    O = Xk.T if transposed else Xk
    rows, cols = W.shape
    scale = update_scale(rows, cols, cfg.scale_coeff)
    W_new = W.astype(np.float64) - float(lr) * scale * O
    if w_is_bf16:
        W_out = round_to_bf16(W_new)
    else:
        W_out = W_new.astype(np.float32)
    return OracleStepResult(W=W_out, M=M_new, O=O, X0=X0, scale=scale)


def muon_step_batch(Ws, Gs, Ms, lrs, cfg: OracleConfig = OracleConfig(), w_is_bf16=None):
    """Independent per-matrix steps over a ragged batch (whole matrices, as in
    the per-expert ownership of tanhow.com's FlexShard paragraph)."""
    out = []
    for i, (W, G, M) in enumerate(zip(Ws, Gs, Ms)):
        bf = bool(w_is_bf16[i]) if w_is_bf16 is not None else False
        out.append(muon_step_matrix(W, G, M, lrs[i], cfg, bf))
    return out

