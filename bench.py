#!/usr/bin/env python3
"""Benchmark of the fp16 TN GEMM  D = C + A.B^T  on GB300.

Headline workload: M=N=K=8192, A and B K-major, fp32 accumulation, fp16
out, C = 0 (uniform [-1,1] operands, seeded).  One step = one gemm_tn call
over that problem (the whole hot path: TMA ring, tcgen05 main loop, C add and
fp16 epilogue).  The metric is TFLOP/s (2*M*N*K per step).

Prints ONE JSON line (rank 0).  Besides the device-timed value it reports:
  e2e           the same metric through the C ABI with host buffers
                (gemm_tn_host): every step copies A, B and C from pinned host
                memory to the device and D back, inside the timed region (row
                panels overlap copies in, GEMMs and copies out; the serial
                one-panel figure beside it)
  roofline      the main kernel against the measured dense bf16/fp16 peak
  cpu_baseline  the CPU oracle (fp64 triple loop) timed on a bounded sample
                of the same workload on this host's cores
  clocks        SM clocks and throttle reasons sampled during the timed region
  extra         other paths, each timed on its own: cuBLAS (torch.addmm) on
                the headline's inputs beside gemm_tn_scaled (context only),
                the skinny M=16 workload's HBM bandwidth, the tiny, square
                (fp16 accumulation) and ragged workloads against both
                rooflines, 4096^3 with K+1 leading dimensions (strided
                route), stream-K against the unsplit kernel, the scaled and
                batched entry point, and the 128-row kernel's K split on
                few-tile shapes

Multi-GPU: the GEMM is one problem per GPU here (replicas only): with
torchrun each rank runs the same workload on its own GPU, and the value is
the work of all ranks divided by the slowest rank's time.

--impl reference times the CPU oracle on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fp16 TN GEMM TFLOP/s at 8192³ and % of GB300 dense FP16 tensor peak"
UNIT = "TFLOP/s"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large")
    ap.add_argument("--shape", default="",
                    help="M,N,K: time that K-major fp32-accumulation problem instead of the "
                         "named workload (uniform [-1,1] operands, B ~ N(0,1/K) when M <= 256, "
                         "C = 0), for profiling one kernel on a chosen size")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--all-extras", action="store_true",
                    help="also time cuBLAS on the headline inputs, the strided route, "
                         "stream-K, the scaled/batched form and the tile K splits")
    ap.add_argument("--only-strided", action="store_true",
                    help="time only the general-stride entry point (4096^3, leading "
                         "dimensions K+1 and N+1; both routes) and print its figures, "
                         "for profiling its kernels")
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--stream-k", type=int, default=0,
                    help="256x256 kernel: 0 auto, 1 split any partial last wave, -1 never")
    ap.add_argument("--tile-kernel", type=int, default=0,
                    help="large path: 0 choose, 1 single-CTA 128xN, 2 CTA-pair 256x256, "
                         "3 single-CTA 256x256")
    return ap.parse_args(argv)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------- helpers

def max_over_ranks(values, device):
    """Element-wise maximum of per-rank values over all ranks (the values
    themselves with one rank).  device: where the reduction tensor lives
    ('cuda' for NCCL, 'cpu' for gloo)."""
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t = torch.tensor(list(values), dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return [float(x) for x in t.tolist()]
    return [float(x) for x in values]


def whole_job_tflops(world_size, flops_per_step, steps, max_total_ms):
    """Throughput of the whole job: every rank's work over the slowest rank's
    time (replicas: each rank runs the same problem on its own GPU)."""
    return world_size * flops_per_step * steps / (max_total_ms * 1e-3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Source files that define each kernel (its device code and the PTX it uses).
KERNEL_SOURCES = {
    "gemm_tn_large_kernel": ["gemm_large.cuh", "common.cuh", "ptx.cuh"],
    "gemm_tn_large2_kernel": ["gemm_large2.cuh", "gemm_large.cuh", "common.cuh", "ptx.cuh"],
    "gemm_tn_skinny_kernel": ["gemm_skinny.cuh", "common.cuh", "ptx.cuh"],
    "gemm_tn_skinny_cluster_kernel": ["gemm_skinny_cluster.cuh", "gemm_skinny.cuh", "common.cuh",
                                      "ptx.cuh"],
    "gemm_tn_wide_kernel": ["gemm_wide.cuh", "gemm_large.cuh", "common.cuh", "ptx.cuh"],
}


def kernel_source_hash(kernel_key: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp16_tensor_gb300", "csrc")
    for fn in KERNEL_SOURCES[kernel_key]:
        p = os.path.join(csrc, fn)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_key: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since those counters were taken."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel_key)
    if not e or e.get("source_hash") != kernel_source_hash(kernel_key):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)  # let the first sample land before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t0 - 0.06 <= ts <= t1 + 0.06]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in use if num(p[1]) is not None]
        mx = [num(p[2]) for p in use if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if p[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use),
                "in_timed_region": bool(inside),
                "power_w_max": max((num(p[3]) or 0.0) for p in use)}


_ORACLE_INPUTS = {}


def oracle_inputs(w):
    """Bits of workload w's operands (generated once per process)."""
    if w.name not in _ORACLE_INPUTS:
        import numpy as np
        import torch

        from dense_fp16_tensor_gb300 import workloads as wl

        def bits(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)
        _ORACLE_INPUTS[w.name] = tuple(bits(t) for t in wl.make_inputs(w))
    return _ORACLE_INPUTS[w.name]


def oracle_sample_rate(w, rows: int, nthreads: int):
    """Time the CPU oracle on the first `rows` rows of workload w (fp64 triple loop)."""
    import oracle
    a, b, c = oracle_inputs(w)
    t0 = time.perf_counter()
    oracle.gemm_tn(rows, w.N, w.K, a, w.ldA, w.a_major, b, w.ldB, w.b_major, c, w.ldC,
                   want_f16=True, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return 2.0 * rows * w.N * w.K / dt / 1e12, dt


def cpu_baseline(w, target_s=12.0):
    import oracle
    cores = oracle.default_threads()
    # calibrate on a few rows, then size the sample to about target_s
    probe_rows = max(1, min(w.M, cores))
    rate, dt = oracle_sample_rate(w, probe_rows, cores)
    rows = int(min(w.M, max(probe_rows, probe_rows * target_s / max(dt, 1e-3))))
    rows = max(cores, rows // cores * cores) if rows >= cores else rows
    rate, dt = oracle_sample_rate(w, rows, cores)
    # one thread on a small fixed slice, for the per-core rate
    one_rows = min(w.M, 8)
    one_rate, one_dt = oracle_sample_rate(w, one_rows, 1)
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {w.M} output rows of the {w.M}x{w.N}x{w.K} problem "
                      f"(fp64 triple loop, {rows * w.N} outputs, {dt:.1f} s)",
            "single_core": {"value": one_rate, "unit": UNIT, "cores": 1,
                            "sample": f"first {one_rows} rows on one thread ({one_dt:.1f} s); "
                                      f"the whole problem would take "
                                      f"{one_dt * w.M / one_rows / 3600:.1f} h at this rate"}}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = pick_workload(args)
    cores = oracle.default_threads()
    # size each step to about one second of oracle work
    probe = max(1, min(w.M, cores))
    _, dt = oracle_sample_rate(w, probe, cores)
    rows = int(min(w.M, max(probe, probe * 1.0 / max(dt, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample_rate(w, rows, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_rate(w, rows, cores)
    total = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / total / 1e12
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name} {w.M}x{w.N}x{w.K} fp16 TN, fp32 accumulate",
                   "sample_rows_per_step": rows, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {rows} of {w.M} output rows per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def pick_workload(args):
    """The named workload, or the K-major problem given by --shape."""
    from dense_fp16_tensor_gb300 import workloads as wl
    if not args.shape:
        return wl.WORKLOADS[args.workload]
    M, N, K = (int(x) for x in args.shape.split(","))
    skinny = M <= 256
    return wl.Workload(f"shape_{M}x{N}x{K}", 9, M, N, K, wl.MAJOR_K, K, wl.MAJOR_K, K, N,
                       wl.ACC_F32, "normal" if skinny else "u11",
                       "normal_k" if skinny else "u11", "zero")


def run_ours(args):
    import torch
    import torch.distributed as dist

    import dense_fp16_tensor_gb300 as g
    from dense_fp16_tensor_gb300 import binding as gb
    from dense_fp16_tensor_gb300 import workloads as wl

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g.build()
    gb.lib()
    if args.only_strided:
        print(json.dumps({"strided_4096": bench_strided(dev, torch.cuda.Stream(dev))}), flush=True)
        return 0

    w = pick_workload(args)
    A_st, B_st, C_st = wl.make_inputs(w)
    A, Bm, CD = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    opts = (gb.make_options(tile_n=args.tile_n, tile_kernel=args.tile_kernel,
                            stream_k=args.stream_k)
            if (args.tile_n or args.tile_kernel or args.stream_k) else None)

    def step(a_ptr=None, b_ptr=None, cd_ptr=None):
        st = gb.gemm_tn_ex(w.M, w.N, w.K, a_ptr or A.data_ptr(), w.ldA, w.a_major,
                           b_ptr or Bm.data_ptr(), w.ldB, w.b_major, cd_ptr or CD.data_ptr(),
                           w.ldC, w.accum, sp, opts)
        if st != gb.OK:
            raise gb.GemmTnError(st)
        return gb.gemm_tn_last_launch_count()

    def barrier():
        if ws > 1:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize()
    kernels_run = gb.gemm_tn_last_kernels()

    # ---- device-timed region: K steps, events around every launch
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    launches = 0
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(args.steps):
            launches += step()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    if rank == 0:
        sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1) if rank == 0 else None

    (total_ms,) = max_over_ranks([total_ms], dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(ws, w.flops, args.steps, total_ms)

    # ---- end to end through the C ABI with host buffers: one gemm_tn_host
    # call per step, A, B and C read from page-locked host memory and D
    # written back to it inside the call.  The library copies B in, then
    # panels of rows of A and C on a copy stream, runs each panel's GEMM as
    # soon as its rows are in and copies its D rows out on a second copy
    # stream; the inputs are declared ready (host_inputs_ready), so each
    # call's copies in follow the previous call's without waiting for its
    # last GEMM and copy out.  The serial form (one panel, calls in stream
    # order: all copies in, the GEMM, the copy out, nothing overlapped) is
    # reported beside it.
    hA = A_st.pin_memory()
    hB = B_st.pin_memory()
    hC = C_st.pin_memory()
    hD = torch.empty_like(C_st).pin_memory()
    h2d = (hA.numel() + hB.numel() + hC.numel()) * 2
    d2h = hD.numel() * 2

    def e2e_run(nsteps, panel_rows, ready):
        o = gb.make_options(tile_n=args.tile_n, tile_kernel=args.tile_kernel,
                            stream_k=args.stream_k, host_panel_rows=panel_rows,
                            host_inputs_ready=ready)
        first = torch.cuda.Event(enable_timing=True)
        last = torch.cuda.Event(enable_timing=True)
        first.record(stream)
        for _ in range(nsteps):
            st = gb.gemm_tn_host(w.M, w.N, w.K, 1.0, hA.data_ptr(), w.ldA, w.a_major,
                                 hB.data_ptr(), w.ldB, w.b_major, 1.0, hC.data_ptr(), w.ldC,
                                 hD.data_ptr(), w.ldC, w.accum, sp, o)
            if st != gb.OK:
                raise gb.GemmTnError(st, "gemm_tn_host")
        last.record(stream)
        torch.cuda.synchronize()
        return first.elapsed_time(last) / nsteps

    e2e_run(2, 0, 1)
    e2e_run(1, w.M, 0)
    barrier()
    e2e_ms = e2e_run(args.e2e_steps, 0, 1)
    e2e_serial_ms = e2e_run(max(2, args.e2e_steps // 2), w.M, 0)
    e2e_ms, e2e_serial_ms = max_over_ranks([e2e_ms, e2e_serial_ms], dev)

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    peaks, peak_kind = load_peaks()
    kernel_ms = statistics.mean(per)
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])  # fp16 dense rate = bf16 dense rate
    path = gb.gemm_tn_plan_path(w.M, w.N, w.K, w.a_major, w.b_major)
    # the dominant kernel of one step, as reported by the library
    kkey = next((k for k in kernels_run.split("+") if k.startswith("gemm_tn")), "").split("<")[0]
    traffic = traffic_for(kkey, w.name) if kkey in KERNEL_SOURCES else None
    if path == gb.PATH_LARGE:
        sustained = float(peaks.get("bf16_tflops_sustained", 0.0)) or None
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "kernel": kernels_run,
                    "peak_kind": f"{peak_kind} bf16 dense burst (fp16 dense rate is equal)",
                    "peak_sustained": sustained,
                    "frac_of_sustained": achieved / sustained if sustained else None,
                    "algorithmic_flops_per_launch": w.flops}
    else:
        gbs = w.min_bytes / (kernel_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]),
                    "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]), "traffic": traffic,
                    "kernel": kernels_run, "peak_kind": peak_kind,
                    "algorithmic_bytes_per_launch": w.min_bytes}

    # The other workloads of the parity set are timed by default (skinny M=16
    # against HBM, tiny / square1024 / ragged against both rooflines); the
    # remaining paths only with --all-extras, so that the line stays short.
    extra = {}
    if not args.no_extra and w.name != "skinny":
        extra["skinny_m16"] = bench_skinny(dev, stream)
        extra["configs"] = bench_configs(dev, stream)
        if args.all_extras:
            if w.name == "large":
                extra["cublas_same_inputs"] = bench_cublas(dev, stream, w, A, Bm,
                                                           steps=max(20, min(400, args.steps)))
            extra["strided_4096"] = bench_strided(dev, stream)
            extra["stream_k_3072x4096x4096"] = bench_stream_k(dev, stream)
            extra["scaled_batched"] = bench_general(dev, stream)
            extra["tile_split_k"] = bench_tile_split(dev, stream)

    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 in, f32 accumulate, f16 out",
        "data": "synthetic (seeded uniform [-1,1] fp16 operands, C = 0)",
        "config": {"workload": f"{w.name}: M={w.M} N={w.N} K={w.K} TN GEMM, "
                               f"A {'K' if w.a_major == 0 else 'M'}-major ld {w.ldA}, "
                               f"B {'K' if w.b_major == 0 else 'N'}-major ld {w.ldB}, "
                               f"{'fp32' if w.accum == 0 else 'fp16'} accumulate, fp16 C/D in place",
                   "M": w.M, "N": w.N, "K": w.K, "parallelism": f"replicas x{ws}",
                   "l2": (f"inputs larger than L2 (A+B+C/D = {w.min_bytes / 2**20:.0f} MiB "
                          "> 129 MB), no flush" if w.min_bytes > 129e6 else
                          "inputs smaller than L2, no flush"),
                   "path": "large" if path == gb.PATH_LARGE else "skinny"},
        "e2e": {"value": whole_job_tflops(ws, w.flops, 1, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": args.e2e_steps,
                "pipelining": "gemm_tn_host (host_inputs_ready): B in, then row panels of "
                              "A and C in on a copy stream, each panel's GEMM on the compute "
                              "stream, its D rows out on a second copy stream; consecutive "
                              "calls overlap",
                "serial_ms_per_step": e2e_serial_ms,
                "h2d_gb_per_s": h2d / (e2e_ms * 1e-3) / 1e9,
                "serial_value": whole_job_tflops(ws, w.flops, 1, e2e_serial_ms)},
        "gpu_launches": launches,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "kernel_ms": {"mean": kernel_ms, "min": min(per), "median": statistics.median(per)},
        "extra": extra,
    }
    # last key on purpose: a short per-workload digest that survives when
    # only the end of the line is kept
    out["configs_summary"] = configs_summary(w, kernel_ms, kernels_run, roofline, extra,
                                             peaks, peak_kind)
    print(json.dumps(out), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def bench_cublas(dev, stream, w, A, Bm, steps=400, rounds=2):
    """Context, not the product path: the headline problem with the same A and
    B, D = A.B^T + C with a separate D and a uniform [-1,1] C, through
    gemm_tn_scaled and through cuBLAS (torch.addmm), timed in alternating
    blocks of back-to-back calls.  Both sit at the board's power limit on
    these operands, so the ratio compares energy per FLOP as much as kernels."""
    import torch

    from dense_fp16_tensor_gb300 import binding as gb
    from dense_fp16_tensor_gb300 import workloads as wl
    M, N, K = w.M, w.N, w.K
    C = wl.draw((M * N,), "u11", 7301).to(dev).view(M, N)
    D = torch.empty_like(C)
    A2, B2 = A.view(M, K), Bm.view(N, K)
    sp = stream.cuda_stream

    def ours():
        st = gb.gemm_tn_scaled(M, N, K, 1.0, A.data_ptr(), K, 0, Bm.data_ptr(), K, 0, 1.0,
                               C.data_ptr(), N, D.data_ptr(), N, gb.ACC_F32, sp)
        if st != gb.OK:
            raise gb.GemmTnError(st)

    def cublas():
        torch.addmm(C, A2, B2.t(), out=D)

    def timed(fn):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    with torch.cuda.stream(stream):
        for _ in range(3):
            ours()
            cublas()
    torch.cuda.synchronize()
    t = {"ours": [], "cublas": []}
    for _ in range(rounds):
        t["ours"].append(timed(ours))
        t["cublas"].append(timed(cublas))
    fl = 2.0 * M * N * K
    out = {"workload": f"M=N=K={M}, D = A.B^T + C (separate D), fp32 accumulate, "
                       f"{rounds} alternating blocks of {steps} calls",
           "cublas_entry": "torch.addmm (cuBLAS)"}
    for k, v in t.items():
        ms = statistics.median(v)
        out[k] = {"ms_per_call": ms, "TFLOP_per_s": fl / (ms * 1e-3) / 1e12}
    out["ratio_ours_over_cublas"] = out["ours"]["TFLOP_per_s"] / out["cublas"]["TFLOP_per_s"]
    del C, D
    return out


def bench_skinny(dev, stream, steps=200):
    """Skinny M=16 workload: achieved HBM GB/s of the split-K path (the 512 MiB
    B operand is larger than L2, so no flush is needed between calls)."""
    import torch

    from dense_fp16_tensor_gb300 import binding as gb
    from dense_fp16_tensor_gb300 import workloads as wl
    w = wl.WORKLOADS["skinny"]
    A_st, B_st, C_st = wl.make_inputs(w)
    A, Bm, CD = A_st.to(dev), B_st.to(dev), C_st.to(dev)
    sp = stream.cuda_stream

    def step():
        st = gb.gemm_tn(w.M, w.N, w.K, A.data_ptr(), w.ldA, 0, Bm.data_ptr(), w.ldB, 0,
                        CD.data_ptr(), w.ldC, 0, sp)
        if st != gb.OK:
            raise gb.GemmTnError(st)
    with torch.cuda.stream(stream):
        for _ in range(5):
            step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    peaks, kind = load_peaks()
    gbs = w.min_bytes / (ms * 1e-3) / 1e9
    return {"workload": "M=16 N=K=16384 fp32 accumulate", "ms_per_call": ms,
            "algorithmic_bytes": w.min_bytes, "GB_per_s": gbs,
            "hbm_peak_GB_per_s": float(peaks["hbm_gbs"]),
            "frac": gbs / float(peaks["hbm_gbs"]), "peak_kind": kind,
            "kernels": gb.gemm_tn_last_kernels(),
            "launches_per_call": gb.gemm_tn_last_launch_count(), "calls": steps,
            "l2": "B (512 MiB) larger than L2, calls back to back"}


def bench_configs(dev, stream, steps=50):
    """The other workloads of the parity set, each through gemm_tn on its own
    layout: tiny (latency), square 1024^3 with fp16 accumulation and ragged
    4000x3000x2500 with an M-major A.  Their inputs fit in L2, so they are
    timed two ways:
      isolated  a 256 MiB buffer is written between calls and every call is
                timed on its own with events (the flush is outside the timed
                spans): one cold call, launch latency included;
      stream    calls back to back over enough copies of the inputs that
                together exceed L2 (each call reads operands no earlier call
                left in L2), timed as a block: per-call time when a stream
                of such GEMMs runs (tiny is latency only and has no stream
                figure)."""
    import torch

    from dense_fp16_tensor_gb300 import binding as gb
    from dense_fp16_tensor_gb300 import workloads as wl
    peaks, kind = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    sp = stream.cuda_stream
    out = {}
    for name in ("tiny", "square1024", "ragged"):
        w = wl.WORKLOADS[name]
        A_st, B_st, C_st = wl.make_inputs(w)
        set_bytes = 2 * (A_st.numel() + B_st.numel() + C_st.numel())
        nsets = 1 if name == "tiny" else max(2, -(-int(160e6) // set_bytes))
        sets = [(A_st.to(dev), B_st.to(dev), C_st.to(dev)) for _ in range(nsets)]
        torch.cuda.synchronize()

        def step(i=0):
            A, Bm, CD = sets[i % nsets]
            st = gb.gemm_tn(w.M, w.N, w.K, A.data_ptr(), w.ldA, w.a_major, Bm.data_ptr(), w.ldB,
                            w.b_major, CD.data_ptr(), w.ldC, w.accum, sp)
            if st != gb.OK:
                raise gb.GemmTnError(st)
        with torch.cuda.stream(stream):
            for i in range(max(5, nsets)):
                step(i)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        with torch.cuda.stream(stream):
            for e0, e1 in ev:
                flush.fill_(1)
                e0.record(stream)
                step()
                e1.record(stream)
        torch.cuda.synchronize()
        ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
        row = {"M": w.M, "N": w.N, "K": w.K,
               "accumulate": "fp16" if w.accum == gb.ACC_F16 else "fp32",
               "a_major": "M" if w.a_major == gb.MAJOR_MN else "K",
               "kernels": gb.gemm_tn_last_kernels()}
        row.update(_rates(w, ms, peaks, ""))
        if nsets > 1:
            calls = 10 * nsets
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for i in range(calls):
                    step(i)
                e1.record(stream)
            torch.cuda.synchronize()
            row.update(_rates(w, e0.elapsed_time(e1) / calls, peaks, "stream_"))
            row["stream_sets"] = nsets
        out[name] = row
        del sets
    # the same isolated timing of a one-element torch kernel: the launch and
    # event floor under which no isolated call can go
    one = torch.zeros(1, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            flush.fill_(1)
            e0.record(stream)
            one.add_(1.0)
            e1.record(stream)
    torch.cuda.synchronize()
    out["floor_us"] = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3
    out["l2"] = ("isolated: 256 MiB written between calls, each call timed alone (median of "
                 f"{steps}); stream: back to back over input copies totalling > 160 MB; "
                 "floor_us: a one-element kernel timed the isolated way")
    out["peak_kind"] = kind
    return out


def _rates(w, ms, peaks, prefix):
    """Per-call time of workload w and its rates against both rooflines."""
    tflops = w.flops / (ms * 1e-3) / 1e12
    gbs = w.min_bytes / (ms * 1e-3) / 1e9
    return {prefix + "us_per_call": ms * 1e3, prefix + "TFLOP_per_s": tflops,
            prefix + "frac_of_tensor_peak": tflops / float(peaks["bf16_tflops"]),
            prefix + "GB_per_s_algorithmic": gbs,
            prefix + "frac_of_hbm_peak": gbs / float(peaks["hbm_gbs"])}


def _short(kernels: str) -> str:
    """Kernel list without the common prefix and suffix."""
    return "+".join(k.replace("gemm_tn_", "").replace("_kernel", "")
                    for k in kernels.split("+") if k)


def configs_summary(w, kernel_ms, kernels_run, roofline, extra, peaks, peak_kind):
    """One short entry per workload of the parity set: time per call, the
    rate against the roofline that bounds it, its fraction, the kernels."""
    r3 = lambda x: None if x is None else round(float(x), 3)  # noqa: E731
    s = {"peaks": f"{peak_kind}: {float(peaks['bf16_tflops'])} TFLOP/s dense, "
                  f"{float(peaks['hbm_gbs'])} GB/s copy"}
    head = {"us": round(kernel_ms * 1e3, 1), roofline["unit"]: round(roofline["achieved"], 1),
            "frac": r3(roofline["frac"]), "bound": roofline["bound"],
            "kernel": _short(kernels_run)}
    sk = extra.get("skinny_m16")
    if sk:
        s["skinny"] = {"us": round(sk["ms_per_call"] * 1e3, 1), "GB/s": round(sk["GB_per_s"], 1),
                       "frac": r3(sk["frac"]), "bound": "hbm", "kernel": _short(sk["kernels"])}
    cf = extra.get("configs", {})
    if "floor_us" in cf:
        s["isolated_floor_us"] = round(cf["floor_us"], 1)
    for name, bound in (("tiny", "latency"), ("square1024", "tensor"), ("ragged", "tensor")):
        c = cf.get(name)
        if not c:
            continue
        e = {"us": round(c["us_per_call"], 1)}
        if bound == "tensor":
            e["TFLOP/s"] = round(c["TFLOP_per_s"], 1)
            e["frac"] = r3(c["frac_of_tensor_peak"])
            if "stream_us_per_call" in c:
                e["stream_us"] = round(c["stream_us_per_call"], 1)
                e["stream_frac"] = r3(c["stream_frac_of_tensor_peak"])
        e["bound"] = bound
        e["kernel"] = _short(c["kernels"])
        s[name] = e
    s[w.name] = head
    return s


def bench_strided(dev, stream, steps=20):
    """General-stride entry point (gemm_tn_strided) on M=N=K=4096 with
    leading dimensions K+1 for A and B and N+1 for C/D (rows TMA cannot
    address), fp32 accumulation: the automatic route (repacking A and B,
    C/D read and written in place) and the copy-producer kernel (no
    workspace), calls back to back."""
    import torch

    from dense_fp16_tensor_gb300 import binding as gb
    from dense_fp16_tensor_gb300 import workloads as wl
    M = N = K = 4096
    ld = K + 1
    A = wl.draw((M * ld,), "u11", 7001).to(dev)
    Bm = wl.draw((N * ld,), "u11", 7002).to(dev)
    CD = torch.zeros(M * (N + 1), dtype=torch.float16, device=dev)
    sp = stream.cuda_stream
    peaks, kind = load_peaks()

    def timed(route, n):
        def step():
            st = gb.gemm_tn_strided_ex(M, N, K, A.data_ptr(), ld, 1, Bm.data_ptr(), ld, 1,
                                       CD.data_ptr(), N + 1, 1, 0, sp, {"path": route})
            if st != gb.OK:
                raise gb.GemmTnError(st)
        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                step()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        return {"kernels": gb.gemm_tn_last_kernels(),
                "launches": gb.gemm_tn_last_launch_count(), "ms_per_call": ms,
                "TFLOP_per_s": tf, "frac_of_peak": tf / float(peaks["bf16_tflops"]),
                "peak_kind": kind}
    out = {"workload": "M=N=K=4096, ld = K+1 (A, B), ldC = N+1, fp32 accumulate"}
    out.update(timed(gb.PATH_AUTO, steps))
    out["copy_route"] = timed(gb.PATH_STRIDED_COPY, max(2, steps // 10))
    return out


def bench_stream_k(dev, stream, steps=50, rounds=3):
    """Stream-K split of the 256 x 256 tile kernel against the unsplit kernel on
    M=3072 N=4096 K=4096 (192 tiles: one full wave of 152 plus 40), fp32
    accumulation; the two are timed in alternating rounds."""
    import torch

    from dense_fp16_tensor_gb300 import binding as gb
    from dense_fp16_tensor_gb300 import workloads as wl
    M, N, K = 3072, 4096, 4096
    A = wl.draw((M * K,), "u11", 7101).to(dev)
    Bm = wl.draw((N * K,), "u11", 7102).to(dev)
    CD = torch.zeros(M * N, dtype=torch.float16, device=dev)
    sp = stream.cuda_stream
    kernels = {}

    def step(sk):
        st = gb.gemm_tn_ex(M, N, K, A.data_ptr(), K, 0, Bm.data_ptr(), K, 0, CD.data_ptr(), N, 0,
                           sp, {"path": gb.PATH_LARGE, "tile_kernel": gb.TILE_WIDE,
                                "stream_k": sk})
        if st != gb.OK:
            raise gb.GemmTnError(st)
        kernels[sk] = gb.gemm_tn_last_kernels()

    def timed(sk):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                step(sk)
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    with torch.cuda.stream(stream):
        for sk in (1, -1, 1, -1):
            step(sk)
    torch.cuda.synchronize()
    t = {1: [], -1: []}
    for _ in range(rounds):
        for sk in (1, -1):
            t[sk].append(timed(sk))
    fl = 2.0 * M * N * K
    ms_sk, ms_plain = statistics.median(t[1]), statistics.median(t[-1])
    return {"workload": "M=3072 N=4096 K=4096 (192 tiles of 256x256 on 152 SMs), fp32 accumulate",
            "stream_k": {"kernels": kernels[1], "ms_per_call": ms_sk,
                         "TFLOP_per_s": fl / (ms_sk * 1e-3) / 1e12},
            "unsplit": {"kernels": kernels[-1], "ms_per_call": ms_plain,
                        "TFLOP_per_s": fl / (ms_plain * 1e-3) / 1e12},
            "speedup": ms_plain / ms_sk}


def bench_tile_split(dev, stream, steps=100):
    """K split on shapes whose tiles leave most SMs idle: the tile path's
    automatic choice (the 128-row kernel's split, or for 1024^2 x 16384 the
    CTA pair's, with the reduction) against the same kernel unsplit; fp32
    accumulation.  (M = 256 with this N would otherwise take the skinny
    path.)"""
    import torch

    from dense_fp16_tensor_gb300 import binding as gb
    from dense_fp16_tensor_gb300 import workloads as wl
    out = {}
    for M, N, K, unsplit in ((512, 512, 8192, {"tile_kernel": 1, "tile_n": 128}),
                             (256, 1024, 16384, {"tile_kernel": 1, "tile_n": 128}),
                             (1024, 1024, 8192, {"tile_kernel": 1, "tile_n": 128}),
                             (1024, 1024, 16384, {"tile_kernel": 2})):
        A = wl.draw((M * K,), "u11", 7301).to(dev)
        Bm = wl.draw((N * K,), "u11", 7302).to(dev)
        CD = torch.zeros(M * N, dtype=torch.float16, device=dev)
        sp = stream.cuda_stream
        row = {}
        for name, opts in (("split", {"path": gb.PATH_LARGE}),
                           ("unsplit", dict(path=gb.PATH_LARGE, **unsplit))):
            def step():
                st = gb.gemm_tn_ex(M, N, K, A.data_ptr(), K, 0, Bm.data_ptr(), K, 0, CD.data_ptr(),
                                   N, 0, sp, opts)
                if st != gb.OK:
                    raise gb.GemmTnError(st)
            with torch.cuda.stream(stream):
                for _ in range(3):
                    step()
            torch.cuda.synchronize()
            kernels = gb.gemm_tn_last_kernels()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(steps):
                    step()
                e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) / steps * 1e3
            row[name] = {"kernels": kernels, "us_per_call": us,
                         "TFLOP_per_s": 2.0 * M * N * K / (us * 1e-6) / 1e12}
        row["speedup"] = row["unsplit"]["us_per_call"] / row["split"]["us_per_call"]
        out[f"{M}x{N}x{K}"] = row
    return out


def bench_general(dev, stream, steps=20):
    """The scaled and batched entry point (gemm_tn_batched): D = alpha A.B^T +
    beta C with a separate D at 8192^3, and two batches of smaller problems
    (64 of 1024^3; 256 of 512^3 with beta = 0), fp32 accumulation, K-major
    operands, calls back to back."""
    import torch

    from dense_fp16_tensor_gb300 import binding as gb
    from dense_fp16_tensor_gb300 import workloads as wl
    peaks, kind = load_peaks()
    out = {}
    for name, M, N, K, L, alpha, beta in (("scaled_8192", 8192, 8192, 8192, 1, 0.5, 2.0),
                                          ("batched_64x1024", 1024, 1024, 1024, 64, 1.0, 1.0),
                                          ("batched_256x512", 512, 512, 512, 256, 1.0, 0.0)):
        A = wl.draw((L * M * K,), "u11", 7201).to(dev)
        Bm = wl.draw((L * N * K,), "u11", 7202).to(dev)
        C = wl.draw((L * M * N,), "u11", 7203).to(dev)
        D = torch.empty(L * M * N, dtype=torch.float16, device=dev)
        sp = stream.cuda_stream

        def step():
            st = gb.gemm_tn_batched(M, N, K, L, alpha, A.data_ptr(), K, M * K, 0, Bm.data_ptr(),
                                    K, N * K, 0, beta, C.data_ptr(), N, M * N, D.data_ptr(), N,
                                    M * N, 0, sp)
            if st != gb.OK:
                raise gb.GemmTnError(st)
        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                step()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        tf = 2.0 * L * M * N * K / (ms * 1e-3) / 1e12
        # compulsory bytes: A and B read once, C read when beta != 0, D written
        nbytes = 2 * L * (M * K + N * K + (M * N if beta != 0.0 else 0) + M * N)
        gbs = nbytes / (ms * 1e-3) / 1e9
        f_t = tf / float(peaks["bf16_tflops"])
        f_h = gbs / float(peaks["hbm_gbs"])
        # FLOP per byte against the ridge point of the two measured peaks
        intensity = 2.0 * L * M * N * K / nbytes
        ridge = float(peaks["bf16_tflops"]) * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
        out[name] = {"M": M, "N": N, "K": K, "batch": L, "alpha": alpha, "beta": beta,
                     "kernels": gb.gemm_tn_last_kernels(), "ms_per_call": ms,
                     "TFLOP_per_s": tf, "frac_of_peak": f_t,
                     "GB_per_s_algorithmic": gbs, "frac_of_hbm_peak": f_h,
                     "flop_per_byte": intensity, "ridge_flop_per_byte": ridge,
                     "bound": "hbm" if intensity < ridge else "tensor",
                     "frac_of_bound": f_h if intensity < ridge else f_t,
                     "peak_kind": kind}
        del A, Bm, C, D
    return out


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
