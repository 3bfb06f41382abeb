"""Seeded synthetic workloads shaped like the pages' weight matrices.

This module only draws random inputs; it holds none of the Muon arithmetic and
is the one piece of code that both the CUDA path's tests/bench and the CPU
oracle use.  Shapes come from the pages: the expert FFN matrix 2048 x 8192 and
the attention projection 7680 x 7680 ("ZAYA1 MoE training on MI300X",
hotelren.com/news/3048137, section 2.1), 16 experts per layer at hidden 2048
(jsqmd.com/news/1098463, section 2), 128 experts of FFN width 8192
(lpnh.cn/news/2841998, section 2.1) and hidden size 6144
(tanhow.com, the activation-offload paragraph).

Every matrix is generated independently from its own seed, so a sample of a
batch can be regenerated on its own.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class MatrixSpec:
    rows: int
    cols: int
    count: int
    kind: str = "gauss"          # "gauss": G ~ N(0,1)*g_scale; "svd": U diag(s) V^T
    g_scale: float = 1.0
    log10_lo: float = -4.0       # for "svd": s = 10**U(log10_lo, 0)
    w_dtype: str = "bf16"        # "bf16" or "f32"


@dataclass(frozen=True)
class Workload:
    name: str
    specs: tuple
    lr: float = 2e-4
    seed_base: int = 0
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def shapes(self):
        out = []
        for s in self.specs:
            out += [(s.rows, s.cols)] * s.count
        return out

    @property
    def n_matrices(self):
        return sum(s.count for s in self.specs)


WORKLOADS = {
    # one 256 x 512 fp32 gradient, seed 0, fp32 weights
    "single_256x512": Workload("single_256x512", (MatrixSpec(256, 512, 1, "gauss", 1.0, w_dtype="f32"),), seed_base=0),
    # one MoE layer's experts: 16 x (2048 x 8192)
    "experts_16x2048x8192": Workload("experts_16x2048x8192", (MatrixSpec(2048, 8192, 16, "gauss", 1e-3),), seed_base=2000),
    # one dense attention projection with a log-uniform spectrum in [1e-4, 1]
    "dense_7680x7680": Workload("dense_7680x7680", (MatrixSpec(7680, 7680, 1, "svd", log10_lo=-4.0),), seed_base=3000),
    # large sparse-MoE layer: 128 x (2048 x 8192)
    "experts_128x2048x8192": Workload("experts_128x2048x8192", (MatrixSpec(2048, 8192, 128, "gauss", 1e-3),), seed_base=4000),
    # ragged mix at hidden 6144, spectra log-uniform in [1e-5, 1]
    "ragged_h6144": Workload("ragged_h6144", (
        MatrixSpec(6144, 2048, 32, "svd", log10_lo=-5.0),
        MatrixSpec(6144, 6144, 4, "svd", log10_lo=-5.0),
        MatrixSpec(2048, 6144, 8, "svd", log10_lo=-5.0),
    ), seed_base=5000),
    # the pages' other GEMM shapes: the MLP expansion 3072 x 12288
    # (hotelren.com/news/3048137, section 2.1) and the Q projection weight
    # 2048 x 1024 (jsqmd.com/news/1098463, section 3.1)
    "mlp_and_qproj": Workload("mlp_and_qproj", (
        MatrixSpec(3072, 12288, 1, "gauss", 1e-3),
        MatrixSpec(2048, 1024, 4, "gauss", 1e-3),
    ), seed_base=6000),
    # four experts of the same shape: a profiling case that still exceeds L2
    "experts_4x2048x8192": Workload("experts_4x2048x8192", (MatrixSpec(2048, 8192, 4, "gauss", 1e-3),), seed_base=2000),
    # scaled-down versions with the same structure, used by parity tests
    "experts_4x256x1024": Workload("experts_4x256x1024", (MatrixSpec(256, 1024, 4, "gauss", 1e-3),), seed_base=12000),
    "dense_768x768": Workload("dense_768x768", (MatrixSpec(768, 768, 1, "svd", log10_lo=-4.0),), seed_base=13000),
    "ragged_h384": Workload("ragged_h384", (
        MatrixSpec(384, 128, 6, "svd", log10_lo=-5.0),
        MatrixSpec(384, 384, 2, "svd", log10_lo=-5.0),
        MatrixSpec(128, 384, 3, "svd", log10_lo=-5.0),
    ), seed_base=15000),
    # shapes that are not tile multiples (ragged edges, tall and wide, tiny)
    "odd_shapes": Workload("odd_shapes", (
        MatrixSpec(200, 520, 1, "gauss", 1.0),
        MatrixSpec(520, 200, 1, "gauss", 1.0),
        MatrixSpec(136, 136, 1, "svd", log10_lo=-3.0),
        MatrixSpec(8, 24, 1, "gauss", 1.0),
        MatrixSpec(1, 40, 1, "gauss", 1.0),
        MatrixSpec(300, 8, 1, "gauss", 1.0),
        MatrixSpec(264, 1000, 1, "gauss", 1e-3),
    ), seed_base=16000),
    # more shape groups than one Newton-Schulz launch takes (21 > 16) and more
    # matrices than one momentum launch takes (70 > 64): every phase runs as a
    # chain of launches
    "many_groups": Workload("many_groups", tuple(
        MatrixSpec(8 + 8 * k, 3 * (8 + 8 * k) + 8, 1, "gauss", 1.0) if k % 2 == 0
        else MatrixSpec(3 * (8 + 8 * k) + 8, 8 + 8 * k, 1, "gauss", 1.0)
        for k in range(20)) + (MatrixSpec(16, 48, 50, "gauss", 1.0),), seed_base=17000),
}

# The workload the throughput metric is quoted on.
HEADLINE = "experts_16x2048x8192"


def matrix_seed(workload: Workload, index: int) -> int:
    return workload.seed_base + index


def _haar(n: int, k: int, gen: torch.Generator, device, dtype) -> torch.Tensor:
    """n x k matrix with orthonormal columns, Haar-distributed: QR of a
    Gaussian matrix with the signs of R's diagonal folded into Q."""
    z = torch.randn(n, k, generator=gen, device=device, dtype=dtype)
    q, r = torch.linalg.qr(z, mode="reduced")
    d = torch.sign(torch.diagonal(r))
    d = torch.where(d == 0, torch.ones_like(d), d)
    return q * d.unsqueeze(0)


def make_matrix(spec: MatrixSpec, seed: int, device="cpu", steady_momentum: bool = False):
    """Returns (W, G, M) for one matrix: W in the spec's dtype, G and M fp32,
    all rows x cols, contiguous, on ``device``.  M is zero unless
    ``steady_momentum`` (then N(0,1) * g_scale, a mid-training state)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    r, c = spec.rows, spec.cols
    if spec.kind == "gauss":
        G = torch.randn(r, c, generator=gen, device=device, dtype=torch.float32) * spec.g_scale
    elif spec.kind == "svd":
        m = min(r, c)
        wdt = torch.float64 if device.type == "cpu" else torch.float32
        U = _haar(r, m, gen, device, wdt)
        V = _haar(c, m, gen, device, wdt)
        u = torch.rand(m, generator=gen, device=device, dtype=wdt)
        s = torch.pow(torch.tensor(10.0, dtype=wdt, device=device), spec.log10_lo * u)
        G = ((U * s.unsqueeze(0)) @ V.T).to(torch.float32)
    else:
        raise ValueError(spec.kind)
    W = torch.randn(r, c, generator=gen, device=device, dtype=torch.float32) * 0.02
    if spec.w_dtype == "bf16":
        W = W.to(torch.bfloat16)
    if steady_momentum:
        M = torch.randn(r, c, generator=gen, device=device, dtype=torch.float32) * spec.g_scale
    else:
        M = torch.zeros(r, c, device=device, dtype=torch.float32)
    return W.contiguous(), G.contiguous(), M.contiguous()


def make_workload(workload: Workload, device="cpu", steady_momentum: bool = False, indices=None):
    """Lists (Ws, Gs, Ms, lrs) for the whole workload, or for ``indices``."""
    Ws, Gs, Ms, lrs = [], [], [], []
    idx = 0
    for spec in workload.specs:
        for _ in range(spec.count):
            if indices is None or idx in indices:
                W, G, M = make_matrix(spec, matrix_seed(workload, idx), device, steady_momentum)
                Ws.append(W)
                Gs.append(G)
                Ms.append(M)
                lrs.append(workload.lr)
            idx += 1
    return Ws, Gs, Ms, lrs


def spec_of(workload: Workload, index: int) -> MatrixSpec:
    idx = 0
    for spec in workload.specs:
        if index < idx + spec.count:
            return spec
        idx += spec.count
    raise IndexError(index)


def symmetric_flops(rows: int, cols: int, iters: int = 5) -> float:
    """FLOPs of one step counting only the upper triangles of the two Gram
    products: per iteration m(m+1)n + m(m+1)m + 2 m^2 n (m = min, n = max)."""
    m, n = min(rows, cols), max(rows, cols)
    return float(iters) * (m * (m + 1) * n + m * (m + 1) * m + 2.0 * m * m * n)


def dense_flops(rows: int, cols: int, iters: int = 5) -> float:
    m, n = min(rows, cols), max(rows, cols)
    return float(iters) * (2.0 * m * m * n + 2.0 * m * m * m + 2.0 * m * m * n)


def workload_flops(workload: Workload, iters: int = 5, symmetric: bool = True) -> float:
    f = symmetric_flops if symmetric else dense_flops
    return sum(f(r, c, iters) for r, c in workload.shapes)

