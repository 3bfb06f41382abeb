"""Per-tile timeline of the tensor-core kernels, from a build with
``-DMUON_TC_TRACE`` (clock64 stamps that the kernels record in device
arrays; nothing is recorded in the default build).

    python -m muon_newton_schulz_gb300.tctrace [--workload NAME] [--steps N]

Builds the traced library into ``_build/trace``, runs warm-up steps and one
traced step of the workload, and prints one JSON object per launch kind
(Gram X X^T, Gram A A^T with the combine, GEMM, GEMM that applies the
update): medians over the leader CTAs of the pairs of

- ``period``: cycles from one tile's accumulator grant to the next;
- ``issue``: from the grant to the tile's last MMA issued (the MMA issuer is
  throttled by the tensor pipe, so this is the pipe's time for the tile);
- ``mma_wait_stages``: cycles the MMA issuer waited for a full ring stage
  per tile, and of those ``mma_wait_first_kblock`` / ``mma_wait_first_4_kblocks``
  on the tile's first one / four k-blocks;
- ``mma_exec``: ``issue - mma_wait_stages``, to compare with the ideal
  (128 cycles per 256 x 256 x 16 CTA-pair MMA);
- ``epi``: the epilogue warp's time from "accumulator full" to "tile done",
  and its waits for prefetched inputs and for staging buffers;
- ``launch_us``: from the first CTA's entry to the last CTA's end
  (%globaltimer, all CTAs), with ``entry_spread_us`` (last entry - first),
  ``setup_us`` (median entry to the end of the grid dependency wait: set-up
  and the wait for the previous kernel), ``work_us`` (median from there to
  the CTA's end) and ``end_spread_us`` (last end - first end);
  ``sm_mhz``: the median CTA's clock64 cycles over its globaltimer time
  from entry to end; ``fill_cycles``: median from the end of the grid
  dependency wait to the first tile's accumulator grant; ``drain_cycles``:
  median from the last tile done to the CTA's end (leader CTAs).

The stamps of the last launch of each kind are kept; the epilogue wait
counters are summed over the traced step's launches of that kind and divided
by their number here.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os

KINDS = ("gram_xxt", "gram_aa_combine", "gemm", "gemm_apply")
# the kernel's trace arrays: [kind][cta][tile][4] stamps, [kind][cta][6] life,
# [kind][cta][4] epilogue waits, [kind][cta][4] MMA waits
K_KINDS, K_CTAS, K_TILES = 4, 160, 96


def _launches_per_kind(iters: int):
    return (iters, iters, max(iters - 1, 0), 1 if iters else 0)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=None)
    ap.add_argument("--steps", type=int, default=3, help="warm-up steps before the traced one")
    args = ap.parse_args()

    from . import build as _build
    lib_path = _build.build(defines=["MUON_TC_TRACE"], out=os.path.join(_build.BUILD, "trace"))
    os.environ["MUON_GB300_LIBRARY"] = lib_path

    import numpy as np
    import torch

    from . import binding as B
    from . import workloads as wl

    lib = B.load_library()
    read = lib.muon_tc_trace_read
    read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    read.restype = ctypes.c_int
    n_tr = K_KINDS * K_CTAS * K_TILES * 4
    n_small = K_KINDS * K_CTAS
    buf = np.zeros(n_tr + n_small * (6 + 4 + 4), dtype=np.int64)

    dev = torch.device("cuda", 0)
    w = wl.WORKLOADS[args.workload or wl.HEADLINE]
    Ws, Gs, Ms, lrs = wl.make_workload(w, dev, steady_momentum=True)
    ms = B.MuonStep(0)
    for _ in range(args.steps):
        ms.step(Ws, Gs, Ms, lrs)
    torch.cuda.synchronize()
    if read(buf.ctypes.data, buf.nbytes) != 0:      # clears the arrays
        raise RuntimeError("muon_tc_trace_read failed")
    ms.step(Ws, Gs, Ms, lrs)
    torch.cuda.synchronize()
    if read(buf.ctypes.data, buf.nbytes) != 0:
        raise RuntimeError("muon_tc_trace_read failed")
    if ms.check_status() != B.MUON_OK:
        raise RuntimeError("kernel status not OK")
    ms.close()

    tr = buf[:n_tr].reshape(K_KINDS, K_CTAS, K_TILES, 4)
    o = n_tr
    life = buf[o:o + n_small * 6].reshape(K_KINDS, K_CTAS, 6)
    o += n_small * 6
    epi = buf[o:o + n_small * 4].reshape(K_KINDS, K_CTAS, 4)
    o += n_small * 4
    mma = buf[o:o + n_small * 4].reshape(K_KINDS, K_CTAS, 4)
    per_kind = _launches_per_kind(5)
    out = {"workload": w.name}
    for k, name in enumerate(KINDS):
        rows = []
        for c in range(0, K_CTAS, 2):            # leader CTAs of the pairs
            t = tr[k, c]
            n = int(np.count_nonzero(t[:, 0]))
            if n < 2:
                continue
            g0, g1, e0, e1 = t[:n, 0], t[:n, 1], t[:n, 2], t[:n, 3]
            launches = max(per_kind[k], 1)
            lc = life[k, c]
            rows.append({
                "fill_cycles": float(g0[0] - lc[4]),
                "drain_cycles": float(lc[5] - e1[n - 1]),
                "tiles": n,
                "period": float(np.median(np.diff(g0))),
                "issue": float(np.median(g1 - g0)),
                "mma_wait_stages": float(mma[k, c, 2]) / n,
                "mma_wait_first_kblock": float(mma[k, c, 0]) / n,
                "mma_wait_first_4_kblocks": float(mma[k, c, 1]) / n,
                "mma_idle_between_tiles": float(np.median(g0[1:] - g1[:-1])),
                "epi": float(np.median(e1 - e0)),
                "epi_wait_inputs": float(epi[k, c, 0]) / n / launches,
                "epi_wait_staging": float(epi[k, c, 1]) / n / launches,
            })
        if not rows:
            continue
        med = {key: round(float(np.median([r[key] for r in rows])), 1) for key in rows[0]}
        med["mma_exec"] = round(med["issue"] - med["mma_wait_stages"], 1)
        med["leader_ctas"] = len(rows)
        lf = life[k]
        lf = lf[lf[:, 0] != 0]
        if len(lf):
            us = lambda v: round(float(v) / 1e3, 2)
            med["launch_us"] = us(lf[:, 2].max() - lf[:, 0].min())
            med["entry_spread_us"] = us(lf[:, 0].max() - lf[:, 0].min())
            med["setup_us"] = us(np.median(lf[:, 1] - lf[:, 0]))
            med["work_us"] = us(np.median(lf[:, 2] - lf[:, 1]))
            med["end_spread_us"] = us(lf[:, 2].max() - lf[:, 2].min())
            med["ctas"] = int(len(lf))
            mhz = (lf[:, 5] - lf[:, 3]) / np.maximum(lf[:, 2] - lf[:, 0], 1) * 1e3
            med["sm_mhz"] = round(float(np.median(mhz)), 0)
        out[name] = med
    print(json.dumps(out, indent=1))


if __name__ == "__main__":
    main()
