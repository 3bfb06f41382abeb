#!/usr/bin/env python3
"""Throughput of the batched Muon step on one GB300 (or N independent
replicas under torchrun), printed as one JSON line.

A step is one muon_step call over the whole workload: momentum + norm, five
Newton-Schulz iterations (Gram X X^T, Gram A A with the b/c combine, GEMM
with the a X epilogue) and the weight update, for every matrix.  The default
workload is one MoE layer's experts, 16 matrices of 2048 x 8192.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, same metric
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Muon NS-orthogonalised matrices/sec and TFLOP/s (5 iters) vs GB300 BF16 TC peak"
UNIT = "matrices/s"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
KERNEL_SOURCES = ["muon_newton_schulz_gb300/csrc/k_tc.cu", "muon_newton_schulz_gb300/csrc/ptx_sm100.cuh",
                  "muon_newton_schulz_gb300/csrc/muon_internal.h", "muon_newton_schulz_gb300/csrc/launch_util.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--mode", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunk", type=int, default=1)
    ap.add_argument("--e2e-slots", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step in a CUDA graph and time its replays (no per-phase profile)")
    ap.add_argument("--no-phase-profile", action="store_true",
                    help="time the steps without the library's per-phase events, so that the handle "
                         "replays each step as a graph (launch-bound workloads); no phases or roofline")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed, so that
    editing a comment does not count as changing the kernel."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_hash() -> str:
    """First 16 hex digits of the sha256 of the kernel sources' code."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """dram bytes per launch of the GEMM kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kh = kernel_hash()
    for line in open(TRAFFIC_FILE):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
        if kv.get("kernel_hash") == kh and kv.get("workload") == workload and "gemm_bytes_per_launch" in kv:
            return float(kv["gemm_bytes_per_launch"])
    return None


# A timed window at least this long runs the GPU into its power cap the way
# the sustained bf16 measurement (4 s of back-to-back GEMMs) does; a shorter
# one is compared with the burst measurement.
SUSTAINED_WINDOW_S = 2.0


def peaks():
    """(bf16 burst TF/s, bf16 sustained TF/s, HBM GB/s, kind)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        burst = float(d["bf16_tflops"])
        return burst, float(d.get("bf16_tflops_sustained", burst)), float(d["hbm_gbs"]), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def roofline_peak(window_s: float, burst_tf: float, sustained_tf: float, kind: str):
    """(peak TF/s, description) for a timed window of `window_s` seconds: the
    sustained figure from SUSTAINED_WINDOW_S on, the burst one below it."""
    sustained = window_s >= SUSTAINED_WINDOW_S
    peak = sustained_tf if sustained else burst_tf
    desc = (f"{kind} bf16 {'sustained' if sustained else 'burst'} "
            f"(timed window {window_s:.2f} s; sustained from {SUSTAINED_WINDOW_S:.0f} s)")
    return peak, desc


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons, each with its
    own timestamp, so that the summary covers the timed window only."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int, period_ms: int = 25):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        out_dir = os.environ.get("MUON_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")
        self.window = None

    def start(self):
        """Starts sampling and waits (up to 5 s) until the first sample is written."""
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)
        return self

    def mark(self, t_begin: float, t_end: float):
        self.window = (t_begin, t_end)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()
            self.proc = None

    @staticmethod
    def _epoch(ts: str):
        ts = ts.strip()
        frac = 0.0
        if "." in ts:
            ts, f = ts.split(".", 1)
            frac = float("0." + f)
        return time.mktime(time.strptime(ts, "%Y/%m/%d %H:%M:%S")) + frac

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        try:
            rows = [l.strip().split(", ") for l in open(self.path) if l.strip()]
        except Exception:
            return out
        parsed = []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                parsed.append((self._epoch(r[0]), float(r[2]), float(r[3]), float(r[4]),
                               [r[6 + k].strip().lower() == "active" for k in range(4)]))
            except ValueError:
                continue
        if not parsed:
            return out
        sel = parsed
        if self.window is not None:
            b, e = self.window
            sel = [x for x in parsed if b <= x[0] <= e]
            if not sel:   # window shorter than the sampling period: nearest samples
                sel = sorted(parsed, key=lambda x: min(abs(x[0] - b), abs(x[0] - e)))[:2]
        reasons = sorted({self.REASONS[k] for x in sel for k in range(4) if x[4][k]})
        return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_min_mhz": min(x[1] for x in sel),
                "sm_max_mhz": max(x[2] for x in sel), "power_w_median": statistics.median(x[3] for x in sel),
                "reasons": reasons, "samples": len(sel), "period_ms": self.period_ms}


def link_rates(host, dev, reps: int = 3):
    """(H2D GB/s, D2H GB/s): best of `reps` copies of one pinned host tensor
    to the device and back, with CUDA events on the current stream."""
    import torch
    d = torch.empty(host.shape, dtype=host.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    nbytes = host.numel() * host.element_size()
    out = []
    for direction in ("h2d", "d2h"):
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if direction == "h2d":
                d.copy_(host, non_blocking=True)
            else:
                host.copy_(d, non_blocking=True)
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b))
        out.append(nbytes / (best / 1e3) / 1e9)
    return out[0], out[1]


def copy_only_ms(Wh, Gh, Mh, Wd, Gd, Md, dev, reps: int = 2):
    """Wall time (best of `reps`) of one step's copies alone: W, G, M host to
    device on one stream while W, M go device to host on another, the same
    pinned buffers and bytes as an end-to-end step, no kernels.  Overwrites the
    device tensors and the host W, M."""
    import torch
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    best = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(s_in):
            for h, d in zip(Wh + Gh + Mh, Wd + Gd + Md):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            for h, d in zip(Wh + Mh, Wd + Md):
                h.copy_(d, non_blocking=True)
        torch.cuda.synchronize(dev)
        best = min(best, (time.perf_counter() - t0) * 1e3)
    return best


def numa_placement(ptr: int):
    """NUMA nodes holding the pages of the mapping that contains `ptr`
    (/proc/self/numa_maps), e.g. "N0=16384", or None."""
    try:
        best = None
        for line in open("/proc/self/numa_maps"):
            start = int(line.split(" ", 1)[0], 16)
            if start <= ptr and (best is None or start > best[0]):
                best = (start, line)
        if best is None:
            return None
        return " ".join(t for t in best[1].split() if t.startswith("N") and "=" in t) or None
    except Exception:
        return None


def gpu_numa_node(dev_index: int):
    """NUMA node of the GPU's PCI function from sysfs, or None."""
    try:
        import torch
        p = torch.cuda.get_device_properties(dev_index)
        bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        return int(open(f"/sys/bus/pci/devices/{bus}/numa_node").read().strip())
    except Exception:
        return None


def oracle_baseline(workload, n_matrices: int, steps: int, warmup: int):
    """Times the fp64 oracle on whole matrices of the workload (host cores)."""
    import numpy as np
    import oracle.muon_oracle as O
    from muon_newton_schulz_gb300 import workloads as wl
    idxs = list(range(workload.n_matrices))
    cores = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        threads = max(int(i.get("num_threads", 1)) for i in info) if info else cores
    except Exception:
        threads = cores
    times = []
    for s in range(warmup + steps):
        i = idxs[s % len(idxs)]
        W, G, M = wl.make_matrix(wl.spec_of(workload, i), wl.matrix_seed(workload, i), "cpu")
        Wn, Gn, Mn = W.float().numpy(), G.numpy(), M.numpy()
        t0 = time.perf_counter()
        for _ in range(n_matrices):
            O.muon_step_matrix(Wn, Gn, Mn, workload.lr, O.OracleConfig(), w_is_bf16=(W.element_size() == 2))
        dt = time.perf_counter() - t0
        if s >= warmup:
            times.append(dt)
    per_step = sum(times) / len(times)
    return n_matrices / per_step, per_step, threads


def run_reference(args):
    from muon_newton_schulz_gb300 import workloads as wl
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    name = args.workload or wl.HEADLINE
    w = wl.WORKLOADS[name]
    rate, per_step, threads = oracle_baseline(w, 1, args.steps, args.warmup)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "matrices": w.n_matrices, "shapes": sorted(set(w.shapes)),
                   "sample_per_step": "one whole matrix of the workload, fp64 numpy oracle"},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "one whole matrix per step (the oracle on the host cores)"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gb300(args):
    import torch
    from muon_newton_schulz_gb300 import binding as B
    from muon_newton_schulz_gb300 import workloads as wl

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload or wl.HEADLINE
    w = wl.WORKLOADS[name]
    mode = B.MUON_MODE_BF16 if args.mode == "bf16" else B.MUON_MODE_FP32_VALIDATE

    B.load_library(build_if_missing=True)
    # every rank owns whole matrices: its own set, shaped like the workload
    # (another layer's experts), seeded by rank
    if rank:
        w = wl.Workload(w.name, w.specs, lr=w.lr, seed_base=w.seed_base + 100000 * rank)
    Ws, Gs, Ms, lrs = wl.make_workload(w, dev, steady_momentum=True)
    ms = B.MuonStep(local, mode=mode)
    descs, n = ms.descs_from_tensors(Ws, Gs, Ms, lrs)
    ws_bytes = ms.workspace_bytes(descs, n)
    ws = ms.workspace(ws_bytes)
    stream = torch.cuda.current_stream(dev)

    def step():
        st = B.muon_step(ms.h, descs, n, ws.data_ptr(), ws.numel(), stream.cuda_stream)
        if st != B.MUON_OK:
            raise B.MuonError(st, B.muon_last_error_message(ms.h))

    clk = ClockSampler(local).start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if ms.check_status() != B.MUON_OK:
        clk.stop()
        raise RuntimeError("kernel status not OK after warm-up: " + B.muon_last_error_message(ms.h))

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    graph = None
    if args.graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        n_before = B.muon_launch_count(ms.h)
        with torch.cuda.graph(graph, stream=side):
            st = B.muon_step(ms.h, descs, n, ws.data_ptr(), ws.numel(), side.cuda_stream)
            if st != B.MUON_OK:
                raise B.MuonError(st, B.muon_last_error_message(ms.h))
        launches_per_step = B.muon_launch_count(ms.h) - n_before
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
    elif not args.no_phase_profile:
        B.muon_set_profiling(ms.h, True)
        B.muon_read_profile(ms.h)  # clear
    n_launch0 = B.muon_launch_count(ms.h)
    n_graph0 = B.muon_graph_launches(ms.h)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    t_begin = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    barrier()
    time.sleep(2 * clk.period_ms / 1e3)   # let the last samples of the window land
    clk.mark(t_begin, t_end)
    clk.stop()
    launches = B.muon_launch_count(ms.h) - n_launch0 if graph is None else launches_per_step * args.steps
    replays = B.muon_graph_launches(ms.h) - n_graph0 if graph is None else args.steps
    ms_total = e0.elapsed_time(e1)
    st, prof = B.muon_read_profile(ms.h)
    B.muon_set_profiling(ms.h, False)
    if ms.check_status() != B.MUON_OK:
        raise RuntimeError("kernel status not OK after the timed steps: " + B.muon_last_error_message(ms.h))
    ms_step = ms_total / args.steps
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms_step], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_step = float(t.item())

    total_mats = w.n_matrices * world
    value = total_mats / (ms_step / 1e3)
    sym_flops = wl.workload_flops(w)
    dense_flops = wl.workload_flops(w, symmetric=False)
    burst_tf, sustained_tf, hbm_gbs, peak_kind = peaks()
    # the roofline's denominator follows the regime of the timed window
    peak_tf, peak_desc = roofline_peak(ms_total / 1e3, burst_tf, sustained_tf, peak_kind)

    # dominant kernel: the GEMM with the a X epilogue (61% of the flops)
    gemm_flops = sum(2.0 * min(r, c) ** 2 * max(r, c) for r, c in w.shapes)
    traffic = measured_traffic(name)
    phase = None
    gemm_ms = achieved = None
    if prof.steps > 0:   # per-phase events (not recorded inside a CUDA graph)
        gemm_ms = prof.ms[3] / max(1, prof.launches[3])
        achieved = gemm_flops / (gemm_ms / 1e3) / 1e12
        phase = {B.PHASE_NAMES[i]: {"ms_per_step": prof.ms[i] / max(1, prof.steps),
                                    "launches_per_step": prof.launches[i] / max(1, prof.steps)}
                 for i in range(B.MUON_NUM_PHASES)}
        # HBM phases against bandwidth: algorithmic bytes per element
        elems = sum(r * c for r, c in w.shapes)
        k1_bytes = elems * (4 + 4 + 4 + 2 + 2)       # read G, M; write M, X as bf16 hi + lo
        wbytes = 2 if name != "single_256x512" else 4
        k5_bytes = elems * (4 + 2 * wbytes)          # read X (hi + lo); read + write W
        phase["momentum_norm"]["gbs"] = k1_bytes / (phase["momentum_norm"]["ms_per_step"] / 1e3) / 1e9
        phase["momentum_norm"]["frac_of_hbm"] = phase["momentum_norm"]["gbs"] / hbm_gbs
        if phase["apply"]["launches_per_step"] > 0:
            phase["apply"]["gbs"] = k5_bytes / (phase["apply"]["ms_per_step"] / 1e3) / 1e9

    # end to end with the state in pinned host memory, through the library's
    # muon_step_host: every step copies G, W, M in and W, M out, chunks of
    # whole matrices pipelined against the steps of other chunks
    e2e = None
    if not args.no_e2e:
        from muon_newton_schulz_gb300.offload import HostOffloadedMuon
        Wh = [x.cpu().pin_memory() for x in Ws]
        Gh = [x.cpu().pin_memory() for x in Gs]
        Mh = [x.cpu().pin_memory() for x in Ms]
        h2d = sum(x.numel() * x.element_size() for x in Wh + Gh + Mh)
        d2h = sum(x.numel() * x.element_size() for x in Wh + Mh)
        h2d_gbs, d2h_gbs = link_rates(Gh[0], dev)
        off = HostOffloadedMuon(local, chunk=args.e2e_chunk, slots=args.e2e_slots, mode=mode)
        for _ in range(2):
            off.step(Wh, Gh, Mh, lrs)       # warm-up: allocates the staging slots, builds the plans
        torch.cuda.synchronize(dev)
        barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            off.step(Wh, Gh, Mh, lrs)
        torch.cuda.synchronize(dev)
        dt = (time.perf_counter() - t0) / args.e2e_steps
        if off.check_status() != B.MUON_OK:
            raise RuntimeError("kernel status not OK after the end-to-end steps")
        off.close()
        copy_ms = copy_only_ms(Wh, Gh, Mh, Ws, Gs, Ms, dev)
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([dt], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            dt = float(t.item())
        # the link bounds the step from below by the slower direction's bytes
        link_ms = max(h2d / (h2d_gbs * 1e9), d2h / (d2h_gbs * 1e9)) * 1e3
        e2e = {"value": total_mats / dt, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": dt * 1e3,
               "api": "muon_step_host (C ABI): W, G, M in pinned host memory",
               "pipeline": f"chunks of {args.e2e_chunk} matrices, {args.e2e_slots} device slots",
               "link_h2d_gbs": h2d_gbs, "link_d2h_gbs": d2h_gbs, "link_bound_ms_per_step": link_ms,
               "frac_of_link_bound": link_ms / (dt * 1e3),
               "copy_only_ms_per_step": copy_ms, "frac_of_copy_only": copy_ms / (dt * 1e3),
               "host_pages_numa": numa_placement(Gh[0].data_ptr()), "gpu_numa_node": gpu_numa_node(local),
               "host_cpus": len(os.sched_getaffinity(0))}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, per, threads = oracle_baseline(w, 1, 1, 0)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"one whole {w.shapes[0][0]}x{w.shapes[0][1]} matrix of the workload, fp64 numpy, {per:.1f} s"}

    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if mode == B.MUON_MODE_BF16 else "f32", "data": "synthetic",
        "config": {"workload": name, "matrices_per_gpu": w.n_matrices, "shapes": sorted(set(w.shapes)),
                   "ns_iters": 5, "parallelism": f"replicas x{world} (whole matrices per rank)",
                   "l2": "inputs larger than L2: 16 x 2048x8192 fp32 G, M and the 1.07 GB of X (hi, lo) per step"
                   if name == wl.HEADLINE else "see workload sizes"},
        "tflops_symmetric": sym_flops / (ms_step / 1e3) / 1e12 * world,
        "tflops_dense_equivalent": dense_flops / (ms_step / 1e3) / 1e12 * world,
        "frac_of_peak_symmetric": sym_flops / (ms_step / 1e3) / 1e12 / peak_tf,
        "frac_of_burst_peak_symmetric": sym_flops / (ms_step / 1e3) / 1e12 / burst_tf,
        "frac_of_sustained_peak_symmetric": sym_flops / (ms_step / 1e3) / 1e12 / sustained_tf,
        "roofline": {"kernel": "k_ns_tc_pair<GEMM> (gemm_update)", "bound": "tensor", "achieved": achieved,
                     "peak": peak_tf, "peak_kind": peak_desc,
                     "burst_peak": burst_tf, "sustained_peak": sustained_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf if achieved is not None else None,
                     "frac_of_burst": achieved / burst_tf if achieved is not None else None,
                     "frac_of_sustained": achieved / sustained_tf if achieved is not None else None,
                     "traffic": traffic,
                     "algorithmic_flops_per_launch": gemm_flops, "avg_launch_ms": gemm_ms},
        "phases": phase,
        "e2e": e2e,
        "gpu_launches": launches,
        "graph_replays": replays,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    ms.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
