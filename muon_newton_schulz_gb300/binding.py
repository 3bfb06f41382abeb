"""ctypes binding of the C ABI in include/muon.h.

The functions keep the C names and only marshal arguments; every step of the
computation runs in the library's CUDA kernels.  ``MuonStep`` is a small
convenience layer that builds descriptors from torch tensors and owns a
torch-allocated workspace (torch is used for device memory and streams
only).  A missing library raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, byref, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

from . import build as _build

MUON_OK = 0
MUON_ERR_INVALID_ARG = 1
MUON_ERR_UNSUPPORTED = 2
MUON_ERR_WORKSPACE = 3
MUON_ERR_CUDA = 4
MUON_ERR_TIMEOUT = 5

MUON_F32 = 0
MUON_BF16 = 1

MUON_MODE_BF16 = 0
MUON_MODE_FP32_VALIDATE = 1

MUON_NUM_PHASES = 5
PHASE_NAMES = ("momentum_norm", "gram_xxt", "gram_aa_combine", "gemm_update", "apply")


class muon_config(ctypes.Structure):
    _fields_ = [
        ("beta", c_float), ("a", c_float), ("b", c_float), ("c", c_float),
        ("eps", c_float), ("scale_coeff", c_float),
        ("ns_iters", c_int32), ("nesterov", c_int32), ("mode", c_int32),
        ("dampening", c_int32),
    ]


class muon_matrix_desc(ctypes.Structure):
    _fields_ = [
        ("rows", c_int64), ("cols", c_int64),
        ("W", c_void_p), ("w_dtype", c_int32), ("reserved0", c_int32), ("ldw", c_int64),
        ("G", c_void_p), ("ldg", c_int64),
        ("M", c_void_p), ("ldm", c_int64),
        ("lr", c_float), ("reserved1", c_int32),
        ("O_out", c_void_p), ("ldo", c_int64),
    ]


MUON_HOST_W = 1
MUON_HOST_G = 2
MUON_HOST_M = 4
MUON_HOST_O = 8


class muon_host_pipeline(ctypes.Structure):
    _fields_ = [("host_buffers", c_int32), ("chunk_matrices", c_int32), ("slots", c_int32), ("reserved", c_int32)]


class muon_phase_stats(ctypes.Structure):
    _fields_ = [
        ("ms", c_double * MUON_NUM_PHASES),
        ("launches", c_int64 * MUON_NUM_PHASES),
        ("steps", c_int64),
    ]


class MuonError(RuntimeError):
    def __init__(self, status, message=""):
        self.status = status
        super().__init__(f"{muon_status_string(status)}: {message}")


_lib = None


def library_path() -> str:
    """The in-tree library, or the file named by MUON_GB300_LIBRARY (a build
    made with other pipeline-shape macros)."""
    return os.environ.get("MUON_GB300_LIBRARY") or _build.LIB


def load_library(build_if_missing: bool = False):
    """Loads the in-tree shared library (building it first if asked)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing: run muon_newton_schulz_gb300.build.build() first")
        _build.build()
    lib = ctypes.CDLL(path)
    H = c_void_p
    lib.muon_config_default.argtypes = [POINTER(muon_config)]
    lib.muon_config_default.restype = None
    lib.muon_create.argtypes = [POINTER(muon_config), c_int, POINTER(H)]
    lib.muon_workspace_size.argtypes = [H, POINTER(muon_matrix_desc), c_int, POINTER(c_size_t)]
    lib.muon_step.argtypes = [H, POINTER(muon_matrix_desc), c_int, c_void_p, c_size_t, c_void_p]
    lib.muon_check_status.argtypes = [H, c_void_p, c_void_p]
    lib.muon_destroy.argtypes = [H]
    lib.muon_status_string.argtypes = [c_int]
    lib.muon_status_string.restype = c_char_p
    lib.muon_last_error_message.argtypes = [H]
    lib.muon_last_error_message.restype = c_char_p
    lib.muon_set_profiling.argtypes = [H, c_int]
    lib.muon_read_profile.argtypes = [H, POINTER(muon_phase_stats)]
    lib.muon_launch_count.argtypes = [H]
    lib.muon_launch_count.restype = c_int64
    lib.muon_plan_builds.argtypes = [H]
    lib.muon_plan_builds.restype = c_int64
    lib.muon_graph_launches.argtypes = [H]
    lib.muon_graph_launches.restype = c_int64
    lib.muon_host_workspace_size.argtypes = [H, POINTER(muon_matrix_desc), c_int, POINTER(muon_host_pipeline),
                                             POINTER(c_size_t)]
    lib.muon_host_workspace_size.restype = c_int
    lib.muon_step_host.argtypes = [H, POINTER(muon_matrix_desc), c_int, POINTER(muon_host_pipeline), c_void_p,
                                   c_size_t, c_void_p]
    lib.muon_step_host.restype = c_int
    lib.muon_step_noalloc.argtypes = [H, POINTER(muon_matrix_desc), c_int, c_void_p]
    lib.muon_step_noalloc.restype = c_int
    for name in ("muon_create", "muon_workspace_size", "muon_step", "muon_check_status", "muon_destroy",
                 "muon_set_profiling", "muon_read_profile"):
        getattr(lib, name).restype = c_int
    _lib = lib
    return lib


# ---- C functions, same names ---------------------------------------------------

def muon_config_default() -> muon_config:
    cfg = muon_config()
    load_library().muon_config_default(byref(cfg))
    return cfg


def muon_create(cfg: muon_config | None, device: int):
    h = c_void_p()
    st = load_library().muon_create(byref(cfg) if cfg is not None else None, device, byref(h))
    return st, h


def muon_workspace_size(h, descs, n: int):
    nbytes = c_size_t(0)
    st = load_library().muon_workspace_size(h, descs, n, byref(nbytes))
    return st, nbytes.value


def muon_step(h, descs, n: int, ws: int, ws_bytes: int, stream: int) -> int:
    return load_library().muon_step(h, descs, n, c_void_p(ws), ws_bytes, c_void_p(stream))


def muon_step_noalloc(h, descs, n: int, stream: int) -> int:
    """muon_step on the library's fixed device workspace (no allocation)."""
    return load_library().muon_step_noalloc(h, descs, n, c_void_p(stream))


MUON_STATIC_WORKSPACE_BYTES = 64 * 1024 * 1024


def muon_check_status(h, ws, stream: int) -> int:
    """ws None reads the status word of muon_step_noalloc's fixed array."""
    return load_library().muon_check_status(h, c_void_p(ws) if ws else None, c_void_p(stream))


def muon_destroy(h) -> int:
    return load_library().muon_destroy(h)


def muon_status_string(st: int) -> str:
    return load_library().muon_status_string(st).decode()


def muon_last_error_message(h) -> str:
    return load_library().muon_last_error_message(h).decode()


def muon_set_profiling(h, enable: bool) -> int:
    return load_library().muon_set_profiling(h, 1 if enable else 0)


def muon_read_profile(h):
    s = muon_phase_stats()
    st = load_library().muon_read_profile(h, byref(s))
    return st, s


def muon_launch_count(h) -> int:
    return int(load_library().muon_launch_count(h))


def make_pipeline(host_buffers: int, chunk_matrices: int = 1, slots: int = 3) -> muon_host_pipeline:
    pl = muon_host_pipeline()
    pl.host_buffers, pl.chunk_matrices, pl.slots, pl.reserved = int(host_buffers), int(chunk_matrices), int(slots), 0
    return pl


def muon_host_workspace_size(h, descs, n: int, pl: muon_host_pipeline):
    nbytes = c_size_t(0)
    st = load_library().muon_host_workspace_size(h, descs, n, byref(pl), byref(nbytes))
    return st, nbytes.value


def muon_step_host(h, descs, n: int, pl: muon_host_pipeline, ws: int, ws_bytes: int, stream: int) -> int:
    """muon_step on descriptors whose selected buffers are host pointers."""
    return load_library().muon_step_host(h, descs, n, byref(pl), c_void_p(ws), ws_bytes, c_void_p(stream))


def muon_plan_builds(h) -> int:
    return int(load_library().muon_plan_builds(h))


def muon_graph_launches(h) -> int:
    return int(load_library().muon_graph_launches(h))


def make_descs(items):
    """``items``: iterable of dicts with rows, cols, W, w_dtype, ldw, G, ldg, M,
    ldm, lr and optionally O_out, ldo (pointers as ints)."""
    items = list(items)
    arr = (muon_matrix_desc * max(1, len(items)))()
    for i, it in enumerate(items):
        d = arr[i]
        d.rows, d.cols = int(it["rows"]), int(it["cols"])
        d.W, d.w_dtype, d.ldw = it.get("W"), int(it.get("w_dtype", MUON_F32)), int(it.get("ldw", it["cols"]))
        d.G, d.ldg = it.get("G"), int(it.get("ldg", it["cols"]))
        d.M, d.ldm = it.get("M"), int(it.get("ldm", it["cols"]))
        d.lr = float(it.get("lr", 0.0))
        d.O_out, d.ldo = it.get("O_out"), int(it.get("ldo", it["cols"]))
    return arr, len(items)


# ---- torch convenience layer ------------------------------------------------------

class MuonStep:
    """One handle plus a cached workspace; ``step`` runs muon_step on torch
    tensors (device memory owned by torch) on the current stream."""

    def __init__(self, device: int = 0, beta=0.95, a=3.4445, b=-4.7750, c=2.0315, eps=1e-7,
                 scale_coeff=0.2, ns_iters=5, nesterov=False, mode=MUON_MODE_BF16, dampening=False):
        cfg = muon_config_default()
        cfg.beta, cfg.a, cfg.b, cfg.c, cfg.eps, cfg.scale_coeff = beta, a, b, c, eps, scale_coeff
        cfg.ns_iters, cfg.nesterov, cfg.mode = int(ns_iters), 1 if nesterov else 0, int(mode)
        cfg.dampening = 1 if dampening else 0
        st, h = muon_create(cfg, device)
        if st != MUON_OK:
            raise MuonError(st, f"muon_create(device={device})")
        self.h = h
        self.cfg = cfg
        self.device = device
        self._ws = None

    def close(self):
        if self.h:
            muon_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def descs_from_tensors(Ws, Gs, Ms, lrs, Os=None):
        import torch
        items = []
        for i, (W, G, M) in enumerate(zip(Ws, Gs, Ms)):
            for t in (W, G, M):
                if t.dim() != 2 or t.stride(1) != 1:
                    raise ValueError("tensors must be 2-D with unit column stride")
            O = Os[i] if Os is not None else None
            items.append(dict(
                rows=W.shape[0], cols=W.shape[1],
                W=W.data_ptr(), w_dtype=MUON_BF16 if W.dtype == torch.bfloat16 else MUON_F32, ldw=W.stride(0),
                G=G.data_ptr(), ldg=G.stride(0), M=M.data_ptr(), ldm=M.stride(0),
                lr=float(lrs[i]),
                O_out=O.data_ptr() if O is not None else None, ldo=O.stride(0) if O is not None else W.shape[1],
            ))
        return make_descs(items)

    def workspace_bytes(self, descs, n) -> int:
        st, nbytes = muon_workspace_size(self.h, descs, n)
        if st != MUON_OK:
            raise MuonError(st, muon_last_error_message(self.h))
        return nbytes

    def workspace(self, nbytes: int):
        import torch
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=f"cuda:{self.device}")
        return self._ws

    def step_descs(self, descs, n, stream=None):
        import torch
        nbytes = self.workspace_bytes(descs, n)
        ws = self.workspace(nbytes)
        cur = torch.cuda.current_stream(self.device).cuda_stream
        s = stream if stream is not None else cur
        st = muon_step(self.h, descs, n, ws.data_ptr(), ws.numel(), s)
        if st != MUON_OK:
            raise MuonError(st, muon_last_error_message(self.h))
        if s != cur:
            # the workspace belongs to the stream it was allocated on: tell the
            # caching allocator it is also in use on `s`, so that a later
            # replacement does not hand the old block out while `s` still runs
            ws.record_stream(torch.cuda.ExternalStream(s, device=torch.device("cuda", self.device)))
        return st

    def step(self, Ws, Gs, Ms, lrs, Os=None, stream=None):
        descs, n = self.descs_from_tensors(Ws, Gs, Ms, lrs, Os)
        return self.step_descs(descs, n, stream)

    def check_status(self, stream=None):
        import torch
        if self._ws is None:
            return MUON_OK
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        return muon_check_status(self.h, self._ws.data_ptr(), s)
