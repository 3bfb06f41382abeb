"""Builds the shared library ``_build/libmuon_gb300.so`` in-tree with nvcc
for sm_103a only.  Translation units compile in parallel; no cmake.

    python -m muon_newton_schulz_gb300.build [--force] [-v] [-DNAME=VALUE ...] [--out DIR]

``-D`` options are passed to every translation unit (for example the
pipeline shape macros of k_tc.cu); with ``--out`` the objects and the
library go to another directory instead of ``_build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libmuon_gb300.so"
LIB = os.path.join(BUILD, LIB_NAME)
INCLUDE = os.path.join(ROOT, "include")

CUDA_SOURCES = ["k_elementwise.cu", "k_simt_f32.cu", "k_tc.cu", "muon_noalloc.cu"]
CXX_SOURCES = ["muon_api.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return r.returncode, " ".join(cmd), r.stdout


def _stale(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=None, out: str | None = None) -> str:
    """Compiles what changed and links the library; returns its path."""
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    bdir = out or BUILD
    lib = os.path.join(bdir, LIB_NAME)
    os.makedirs(bdir, exist_ok=True)
    defs = [f"-D{d}" for d in (defines or [])]
    if defs:
        force = True
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "muon.h"))
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda, "include"), *defs]
    jobs = []
    objs = []
    for src in CUDA_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc, *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", *common, "-c", s, "-o", o])
    for src in CXX_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc, "-x", "c++", "-Xcompiler", "-fPIC", *common, "-c", s, "-o", o])
    if jobs:
        with ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
            results = list(ex.map(_run, jobs))
        for rc, cmd, text in results:
            if verbose or rc != 0:
                sys.stderr.write(cmd + "\n" + text)
            if rc != 0:
                raise RuntimeError("compilation failed: " + cmd + "\n" + text)
    if force or jobs or _stale(lib, objs):
        tmp = lib + ".tmp"
        rc, cmd, text = _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"])
        if rc != 0:
            raise RuntimeError("link failed: " + cmd + "\n" + text)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    args = sys.argv[1:]
    defines = [a[2:] for a in args if a.startswith("-D")]
    out = args[args.index("--out") + 1] if "--out" in args else None
    print(build(force="--force" in args, verbose="-v" in args, defines=defines, out=out))
