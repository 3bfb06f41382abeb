"""Batched Muon optimizer step (momentum, Frobenius normalisation, five
Newton-Schulz iterations on upper-triangle Gram tiles, scaled weight update)
as hand-written sm_103a CUDA kernels behind a C ABI.

``binding`` marshals arguments to the shared library; ``workloads`` draws the
seeded synthetic inputs.  The library is loaded on first use and its absence
is an error, never a fallback.
"""
from . import binding, workloads  # noqa: F401

__all__ = ["binding", "workloads"]
