#!/usr/bin/env python3
"""Throughput benchmark of the nonuniform FFT hot path on GB300.

One step = one type 1 transform (spread -> FFT -> correct) plus, for
workloads that have one, one type 2 transform (correct/pad -> FFT ->
interpolate) of the workload's M points, each through the C ABI, with the
points already bin-sorted (setpts is excluded, as in the metric).  value =
nonuniform points transformed per second over the whole job: M per transform
per step per GPU.

Prints ONE JSON line (rank 0).  On one GPU the line also carries
"per_workload": the other workloads, a few steps each, with their throughput,
stage times and per-kernel HBM rooflines.  --impl reference times the CPU
oracle (the three-step NUFFT in double precision, on every host core) on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from nonuniform_fft_gb300 import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "2d_f32_N1024_M1e7"
METRIC = "NU points/s (type1 & type2, exec excl. setpts) and % of GB300 HBM roofline"
L2_FLUSH_BYTES = 256 << 20
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "nonuniform_fft_gb300", "csrc")
KERNEL_SOURCES = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                        if f.endswith((".cu", ".cuh")))


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS) + ["all"])
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the other workloads' short measurements (per_workload)")
    ap.add_argument("--per-workload-steps", type=int, default=5)
    ap.add_argument("--sweep", action="store_true",
                    help="time the spreading / interpolation kernel over a grid of plan options "
                         "(bins, M_sub, columns per lane, threads) for --workload, or for every "
                         "workload with --workload all; one JSON line per option set")
    ap.add_argument("--sweep-type", type=int, choices=[1, 2], default=None,
                    help="sweep only the type 1 (spreading) or type 2 (interpolation) plans")
    ap.add_argument("--cpu-sample", type=int, default=0,
                    help="points per transform in the CPU baseline sample (0: auto)")
    ap.add_argument("--sigma", type=float, default=2.0,
                    help="upsampling factor in (1, 2] (nufft_makeplan_upsampled when < 2)")
    ap.add_argument("--batch", type=int, default=1,
                    help="strength vectors per transform (nufft_execute_batch); 1: nufft_execute")
    ap.add_argument("--opt", action="append", default=[], metavar="KEY=VALUE",
                    help="plan option for both plans (nufft_set_opt), e.g. msub=1024; repeatable")
    return ap.parse_args()


def plan_opts(args) -> dict:
    out = {}
    for kv in args.opt:
        k, v = kv.split("=", 1)
        out[k] = float(v)
    return out


# ------------------------------------------------------------------ helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_step: int, steps: int, t_max_s: float) -> float:
    """Whole-job throughput: units every rank processed / slowest rank's time."""
    return world * units_per_step * steps / t_max_s


def algorithmic_bytes(wl: W.Workload, n, nvec: int = 1) -> dict:
    """Minimum bytes each kernel must move per launch of nvec vectors:
    coordinates (d reals) and one 4-byte permutation index per point once,
    and per vector one complex strength / result per point plus the
    fine-grid traffic."""
    cs = 4 if wl.dtype == "f32" else 8
    cb = 2 * cs
    d = wl.dim
    M = wl.M
    cells = int(np.prod(n))
    modes = int(np.prod(wl.N))
    v = nvec
    return {
        "spread": M * (d * cs + 4) + v * (M * cb + 2 * cells * cb),  # points; c in; grid read + written
        "interp": M * (d * cs + 4) + v * (cells * cb + M * cb),      # points; grid in, c out
        "deconv": v * 2 * modes * cb,
        "pad": v * (modes * cb + cells * cb),
    }


# ALU roofline of the spreading and interpolation kernels: each point adds
# (or gathers) w^d complex values times a real weight, 2 w^d real
# multiply-adds.  Peaks from the unit counts and clocks: FP32, 128 FMA lanes
# per SM x 152 SMs x 2.07 GHz; FP64, the nominal 1.25 TFLOP/s of this part
# (the double-precision kernels run two-float arithmetic on the FP32 pipes,
# so they are measured against the FP64 rate they stand in for).
FP32_TFMA = 128 * 152 * 2.07e9 / 1e12
FP64_TFMA = 1.25 / 2


def alu_roofline(wl: W.Workload, w: int, launch_ms: float, vpp: int = 1) -> dict:
    fma = 2.0 * w ** wl.dim * wl.M * vpp
    achieved = fma / (launch_ms / 1e3) / 1e12
    peak = FP32_TFMA if wl.dtype == "f32" else FP64_TFMA
    return {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFMA/s",
            "frac": achieved / peak, "algorithmic_fma_per_launch": fma,
            "peak_source": ("FP32: 128 lanes x 152 SMs x 2.07 GHz" if wl.dtype == "f32"
                            else "FP64: nominal 1.25 TFLOP/s (two-float kernels on the FP32 pipes)")}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources."""
    try:
        with open(TRAFFIC_PATH) as fh:
            t = json.load(fh)
    except (OSError, ValueError):
        return None
    e = t.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


_libcuda = None


def reset_l2_priorities():
    """Return the L2 lines that kernels marked evict-last to normal priority
    (cuCtxResetPersistingL2Cache on the current context, which the CUDA
    runtime made current for this thread), so that the flush that follows
    evicts them too.  Returns the driver's status (0 = success)."""
    global _libcuda
    if _libcuda is None:
        import ctypes
        _libcuda = ctypes.CDLL("libcuda.so.1")
    return _libcuda.cuCtxResetPersistingL2Cache()


def flush_l2(flush, stream):
    """Evict the previous step's data from L2 (untimed): demote evict-last
    lines, then write a buffer larger than L2."""
    import torch
    torch.cuda.current_stream().synchronize()
    stream.synchronize()
    rc = reset_l2_priorities()
    if rc != 0:
        raise RuntimeError(f"cuCtxResetPersistingL2Cache failed: {rc}")
    with torch.cuda.stream(stream):
        flush.zero_()


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows]
        smax = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle

# kernel-weighted grid updates (w^d per point and transform) one host thread
# gets through in about a second of the oracle's plain loops
CPU_CELLS_PER_THREAD = 1.2e8


def cpu_sample_points(wl: W.Workload, budget_cells: float, sigma: float = 2.0) -> int:
    """Points per transform in a CPU-oracle sample: about budget_cells
    kernel-weighted grid updates (w^d per point), at most the whole workload."""
    import oracle
    w = oracle.es_params(wl.eps, sigma)[0]
    return int(min(wl.M, max(20000, budget_cells / w ** wl.dim)))


def cpu_oracle_run(wl: W.Workload, sample_M: int, steps: int = 1, sigma: float = 2.0) -> dict:
    """Time the oracle's three-step NUFFT (type 1, plus type 2 when the
    workload has it) on the first sample_M points of the workload, on every
    host core it may use; returns points/s over `steps` repeats."""
    import oracle
    sub = wl.scaled(M=sample_M)
    pts, c = W.sample(sub)
    fk = W.coefficients(wl)
    oracle.build()
    cores = oracle.cpu_threads()
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.nufft_type1(pts, c, wl.N, wl.eps, wl.iflag[1], sigma, threads=cores)
        if 2 in wl.types:
            oracle.nufft_type2(pts, fk, wl.N, wl.eps, wl.iflag[2], sigma, threads=cores)
    dt = time.perf_counter() - t0
    per_step = sample_M * len(wl.types)
    types = " + ".join(f"type {t}" for t in wl.types)
    whole = "all" if sample_M == wl.M else f"{sample_M} of"
    return {"value": per_step * steps / dt, "unit": "NU points/s", "cores": cores,
            "kind": "oracle", "seconds": dt,
            "sample": f"{whole} {wl.M} points of {wl.name}, full {'x'.join(map(str, wl.N))} "
                      f"modes, {types}, x{steps}; sigma {sigma:g}; double precision; spreading "
                      f"and interpolation on {cores} threads (point chunks), numpy FFT"}


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    cores = oracle.cpu_threads()
    # bounded: about a minute of CPU work for the whole --steps + --warmup run
    per_step = args.cpu_sample or cpu_sample_points(
        wl, cores * CPU_CELLS_PER_THREAD / max(1, (args.steps + args.warmup) / 2), args.sigma)
    per_step = min(per_step, wl.M)
    if args.warmup:
        cpu_oracle_run(wl, min(per_step, 20000), 1, args.sigma)
    r = cpu_oracle_run(wl, per_step, args.steps, args.sigma)
    line = {
        "impl": "reference", "metric": METRIC, "value": r["value"], "unit": "NU points/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * r["seconds"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "N": list(wl.N), "M": wl.M, "eps": wl.eps,
                   "sigma": args.sigma, "sample_points_per_transform": per_step},
        "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": r["value"], "unit": "NU points/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def kernel_names(wl: W.Workload, method1: int, method2: int, tile3d: int = 1, igroup: int = 0) -> dict:
    """Names of the spreading and interpolation kernels the plans launch."""
    import nonuniform_fft_gb300 as nf
    df = "_df" if wl.dtype == "f64" else ""
    regtile = {1: "spread_reg1d" + df + "_kernel", 2: "spread_regtile2d_kernel",
               3: "spread_slab3d_kernel" if tile3d == 2 else "spread_plane3d" + df + "_kernel"}[wl.dim]
    spread = {nf.METHOD_SM: "spread_sm_kernel", nf.METHOD_GM_SORT: "spread_gm_kernel",
              nf.METHOD_GM: "spread_gmu_kernel", nf.METHOD_REGTILE: regtile}[method1]
    sm_interp = {1: "interp_sm1d" + df + "_kernel", 2: "interp_sm_kernel",
                 3: "interp_sm3d_df_kernel" if wl.dtype == "f64" else
                 ("interp_group3d_kernel" if igroup >= 2 else "interp_sm3d_bank_kernel")}
    interp = {nf.METHOD_GM_SORT: "interp_gm_kernel", nf.METHOD_GM: "interp_gmu_kernel"}.get(
        method2, sm_interp[wl.dim])
    return {"spread": spread, "interp": interp}


def hbm_peak():
    try:
        with open(PEAKS_PATH) as fh:
            return float(json.load(fh)["hbm_gbs"]), "MEASURED_PEAKS.json hbm_gbs (measured copy bandwidth)"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def measure(wl, args, dev, stream, opts, steps: int, warmup: int, B: int = 1,
            host_legs: bool = True, clocks: bool = False) -> dict:
    """Time `steps` steps (type 1, plus type 2 when the workload has it) of
    one workload with its points already sorted; L2 flushed between steps.
    Returns the throughput, per-stage times, per-kernel HBM rooflines and,
    with host_legs, the end-to-end (host buffers) figure and timing scopes."""
    import torch

    import nonuniform_fft_gb300 as nf

    rank, world, local = dist_env()
    cname = "complex64" if wl.dtype == "f32" else "complex128"
    ctorch = getattr(torch, cname)
    pts, c_np = W.sample(wl)
    fk_np = W.coefficients(wl)
    N = wl.N
    with torch.cuda.stream(stream):
        xs = [torch.from_numpy(p).to(dev) for p in pts]
        # B vectors: the workload's own, then copies rotated by a phase each
        c_in = torch.from_numpy(c_np).to(dev)
        f_in = torch.from_numpy(fk_np).to(dev)
        if B > 1:
            ph = torch.exp(1j * torch.arange(B, dtype=torch.float64, device=dev)).to(ctorch)
            c_in = (ph[:, None] * c_in[None, :]).contiguous()
            f_in = (ph[:, None] * f_in[None, :]).contiguous()
        f_out = torch.empty(B * int(np.prod(N)), dtype=ctorch, device=dev)
        c_out = torch.empty(B * wl.M, dtype=ctorch, device=dev)
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream.synchronize()
    del pts, c_np, fk_np

    has2 = 2 in wl.types
    p1 = nf.Plan(1, N, wl.iflag[1], wl.eps, cname, stream=stream.cuda_stream, sigma=args.sigma,
                 **opts)
    p2 = nf.Plan(2, N, wl.iflag[2], wl.eps, cname, stream=stream.cuda_stream, sigma=args.sigma,
                 **opts) if has2 else None
    try:
        for p in (p1, p2):
            if p is not None:
                p.setpts(*xs)
                p.setpts(*xs)   # the "setpts" scope is this second call: buffers allocated
        info = p1.info()
        info2 = p2.info() if has2 else None
        n = [info["n1"], info["n2"], info["n3"]][: wl.dim]

        def step():
            if B == 1:
                p1.execute(c_in, f_out)
                if has2:
                    p2.execute(c_out, f_in)
            else:
                p1.execute_batch(B, c_in, f_out)
                if has2:
                    p2.execute_batch(B, c_out, f_in)

        for _ in range(warmup):
            step()
        stream.synchronize()

        ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        stage = {k: 0.0 for k in ("spread", "fft1", "deconv", "zero", "pad", "fft2", "interp")}
        zeros = {k: 0.0 for k in nf.TIMING_KEYS}
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        clk = ClockSampler(local) if clocks else None
        if clk:
            clk.__enter__()
        try:
            for i in range(steps):
                flush_l2(flush, stream)                 # evict the inputs from L2 (untimed)
                ev0[i].record(stream)
                step()
                ev1[i].record(stream)
                t1 = p1.timings()                       # waits for this step's events
                t2 = p2.timings() if has2 else zeros
                stage["spread"] += t1["spread_interp"]
                stage["fft1"] += t1["fft"]
                stage["deconv"] += t1["deconv_pad"]
                stage["zero"] += t1["zero"]
                stage["pad"] += t2["deconv_pad"]
                stage["fft2"] += t2["fft"]
                stage["interp"] += t2["spread_interp"]
            torch.cuda.synchronize()
        finally:
            if clk:
                clk.__exit__(None, None, None)
        if world > 1:
            dist.barrier()
        total_ms = sum(a.elapsed_time(b) for a, b in zip(ev0, ev1))
        t_max = reduce_max(total_ms, dev)
        pts_per_step = wl.M * len(wl.types) * B
        value = job_throughput(world, pts_per_step, steps, t_max / 1e3)

        # HBM roofline of the spreading and interpolation kernels (per-launch
        # averages of their CUDA-event times over the timed region)
        vpp = min(B, info["batch"]) if B > 1 else 1       # vectors one launch processes
        launches = -(-B // vpp)                           # spread / interp launches per transform
        algo = algorithmic_bytes(wl, n, vpp)
        peak, peak_source = hbm_peak()
        names = kernel_names(wl, info["method"], info2["method"] if has2 else 0, info.get("tile3d", 1),
                             info2.get("igroup", 0) if has2 else 0)
        rooflines = {}
        for key in (("spread", "interp") if has2 else ("spread",)):
            ms = stage[key] / (steps * launches)
            achieved = algo[key] / (ms / 1e3) / 1e9
            rooflines[key] = {"bound": "hbm", "kernel": names[key], "achieved": achieved,
                              "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                              "traffic": load_traffic(names[key], wl.name),
                              "algorithmic_bytes_per_launch": algo[key], "launch_ms": ms,
                              "peak_source": peak_source,
                              "alu": alu_roofline(wl, info["w"], ms, vpp)}
        dom = max(rooflines, key=lambda k: rooflines[k]["launch_ms"])
        out = {"value": value, "t_max_ms": t_max, "total_ms_rank0": total_ms, "stage": stage,
               "info": info, "n": n, "rooflines": rooflines, "dominant": dom,
               "pts_per_step": pts_per_step, "vpp": vpp, "launches": launches,
               "clocks": clk.summary() if clk else None,
               # per transform and launch pass: spreading or interpolation plus the
               # correction kernel, or plus the two fused FFT passes
               "gpu_launches": (2 if has2 else 1) * (3 if info["fft"] else 2) * launches * steps}
        out["setpts_ms"] = p1.timings()["setpts"] + (p2.timings()["setpts"] if has2 else 0.0)
        if not host_legs:
            return out

        # end to end through the C ABI with pinned host buffers
        hc = c_in.cpu().pin_memory()
        hf = f_in.cpu().pin_memory()
        hf_out = torch.empty(B * int(np.prod(N)), dtype=ctorch).pin_memory()
        hc_out = torch.empty(B * wl.M, dtype=ctorch).pin_memory()

        def host_step():
            # host c in, host f out; host f in, host c out (synchronous calls)
            if B == 1:
                p1.execute(hc, hf_out)
                if has2:
                    p2.execute(hc_out, hf)
            else:
                p1.execute_batch(B, hc, hf_out)
                if has2:
                    p2.execute_batch(B, hc_out, hf)

        host_step()
        e2e_steps = max(3, min(steps, 10))
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_step()
        el = reduce_max(time.perf_counter() - t0, dev)
        cb = hc.element_size()
        modes = int(np.prod(N))
        out["e2e"] = {"value": job_throughput(world, pts_per_step, e2e_steps, el),
                      "unit": "NU points/s",
                      "h2d_bytes_per_step": B * (wl.M * cb + (modes * cb if has2 else 0)),
                      "d2h_bytes_per_step": B * (modes * cb + (wl.M * cb if has2 else 0))}

        # "total+mem" scope: host arrays in and out, setpts and exec, wall clock
        hx = [x.cpu().pin_memory() for x in xs]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        p1.setpts(*hx)
        if has2:
            p2.setpts(*hx)
        host_step()
        torch.cuda.synchronize()
        out["total_mem_ms"] = 1e3 * (time.perf_counter() - t0)
        return out
    finally:
        p1.close()
        if p2 is not None:
            p2.close()


def stage_summary(r: dict, steps: int) -> dict:
    return {k: v / steps for k, v in r["stage"].items()}


def workload_config(wl, args, r, opts, B, world) -> dict:
    info = r["info"]
    return {"workload": wl.name, "dim": wl.dim, "N": list(wl.N), "M": wl.M,
            "eps": wl.eps, "sigma": args.sigma, "w": info["w"], "fine_grid": r["n"],
            "dist": wl.dist, "dtype": wl.dtype,
            "types": " + ".join(f"type {t} (iflag {wl.iflag[t]:+d})" for t in wl.types)
                     + " per step",
            "points_per_step_per_gpu": r["pts_per_step"],
            "bins": [info["bin1"], info["bin2"], info["bin3"]][: wl.dim],
            "msub": info["msub"], "nsub": info["nsub"], "sms": info["sms"],
            "fine_grid_fft": ("fused pruned passes (x and y) with the correction in the y pass; "
                              "stage fft1/fft2 hold both passes, deconv/pad are 0"
                              if info["fft"] else "cuFFT + correction kernel"),
            "l2": "flushed between timed steps (256 MiB write, untimed)",
            "plan_options": opts,
            "vectors_per_transform": B, "vectors_per_launch": r["vpp"],
            "parallelism": f"replicas x{world}"}


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    import nonuniform_fft_gb300 as nf

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    nf.load_library()
    stream = torch.cuda.Stream(dev)
    opts = plan_opts(args)
    B = args.batch
    K = args.steps

    r = measure(wl, args, dev, stream, opts, K, args.warmup, B, host_legs=not args.no_e2e,
                clocks=True)

    # the other workloads: a few steps each, default options, one GPU only
    per_workload = None
    if world == 1 and not args.no_per_workload:
        per_workload = {}
        for name, other in W.WORKLOADS.items():
            if name == wl.name:
                continue
            ro = measure(other, args, dev, stream, {}, args.per_workload_steps, 3, 1,
                         host_legs=False)
            per_workload[name] = {
                "value": ro["value"], "unit": "NU points/s",
                "ms_per_step": ro["t_max_ms"] / args.per_workload_steps,
                "steps": args.per_workload_steps, "warmup": 3,
                "stage_ms_per_step": stage_summary(ro, args.per_workload_steps),
                "setpts_ms": ro["setpts_ms"],
                "roofline": ro["rooflines"][ro["dominant"]],
                "rooflines": ro["rooflines"],
                "gpu_launches": ro["gpu_launches"],
                "config": workload_config(other, args, ro, {}, 1, world),
            }
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        budget = oracle.cpu_threads() * CPU_CELLS_PER_THREAD
        cpu = cpu_oracle_run(wl, args.cpu_sample or cpu_sample_points(wl, budget, args.sigma), 1,
                             args.sigma)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}

    if rank == 0:
        # timing scopes of [cuFINUFFT] Sec. IV-C: "exec" (the step above), "total"
        # (setpts + exec, on the device) and "total+mem" (host arrays in and out,
        # setpts and exec, wall clock, synchronous)
        scopes = {"exec_ms": r["t_max_ms"] / K, "setpts_ms": r["setpts_ms"],
                  "total_ms": r["t_max_ms"] / K + r["setpts_ms"],
                  "setpts_note": "device time of a second setpts per plan (buffers allocated)"}
        if "total_mem_ms" in r:
            scopes["total_mem_ms"] = r["total_mem_ms"]
        line = {
            "metric": METRIC, "value": r["value"], "unit": "NU points/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": r["t_max_ms"] / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic",
            "config": workload_config(wl, args, r, opts, B, world),
            "stage_ms_per_step": stage_summary(r, K),
            "scopes": scopes,
            "step_ms_rank0": r["total_ms_rank0"] / K,
            "roofline": r["rooflines"][r["dominant"]],
            "rooflines": r["rooflines"],
            "cpu_baseline": cpu,
            "e2e": r.get("e2e"),
            "gpu_launches": r["gpu_launches"],
            "clocks": r["clocks"],
            "per_workload": per_workload,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ option sweep

# Option sets swept per workload and transform type (plan options of
# nufft_set_opt; {} is the library's default).  Type 1 plans use the
# register-tile spreader, type 2 plans the shared-memory interpolator.
def sweep_space(wl: W.Workload, t: int) -> list:
    def grid(**axes):
        out = [{}]
        for k, vals in axes.items():
            out = [dict(o, **{k: v}) for o in out for v in vals]
        return out
    if wl.dim == 2 and t == 1:
        return [{}] + grid(regtile_cols=[1, 2], bin2=[32, 64, 128], msub=[256, 512, 1024, 2048])
    if wl.dim == 2 and t == 2:
        return [{}] + [dict(o, bin2=o["bin1"]) for o in
                       grid(bin1=[16, 26, 32, 48], msub=[1024, 2048, 4096], threads=[128, 256, 512])]
    if wl.dim == 3 and t == 1:
        return [{}] + grid(bin2=[4, 8, 16, 32], msub=[2048, 4096, 8192])
    if wl.dim == 3 and t == 2 and wl.dtype == "f32":   # one point per thread, or grouped by window
        return ([{}] + grid(igroup=[1], msub=[2048, 4096, 8192], threads=[256, 512, 1024])
                + grid(igroup=[2, 3, 4], msub=[2048, 4096, 8192], threads=[128, 256]))
    if wl.dim == 3 and t == 2:
        return [{}] + grid(msub=[2048, 4096, 8192], threads=[256, 512, 1024])
    if wl.dim == 1 and t == 1:
        return [{}] + grid(msub=[128, 256, 512, 1024, 2048])
    return [{}] + grid(bin1=[256, 512, 1024, 2048], msub=[512, 1024, 2048, 4096])


def run_sweep(args):
    import torch

    import nonuniform_fft_gb300 as nf

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    nf.load_library()
    stream = torch.cuda.Stream(dev)
    names = sorted(W.WORKLOADS) if args.workload == "all" else [args.workload]
    best = {}
    for name in names:
        wl = W.WORKLOADS[name]
        cname = "complex64" if wl.dtype == "f32" else "complex128"
        ctorch = getattr(torch, cname)
        pts, c_np = W.sample(wl)
        with torch.cuda.stream(stream):
            xs = [torch.from_numpy(p).to(dev) for p in pts]
            c_in = torch.from_numpy(c_np).to(dev)
            f_in = torch.from_numpy(W.coefficients(wl)).to(dev)
            f_out = torch.empty(int(np.prod(wl.N)), dtype=ctorch, device=dev)
            c_out = torch.empty(wl.M, dtype=ctorch, device=dev)
            flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        stream.synchronize()
        steps = 3 if wl.dim == 3 and wl.dtype == "f64" else 6
        for t in wl.types:
            if args.sweep_type and t != args.sweep_type:
                continue
            for opts in sweep_space(wl, t):
                try:
                    plan = nf.Plan(t, wl.N, wl.iflag[t], wl.eps, cname, stream=stream.cuda_stream, **opts)
                    plan.setpts(*xs)
                except nf.NufftError as e:      # an option set the kernel cannot take
                    print(json.dumps({"sweep": name, "type": t, "opts": opts, "error": str(e)}), flush=True)
                    continue
                info = plan.info()
                ms = []
                for i in range(2 + steps):
                    flush_l2(flush, stream)
                    if t == 1:
                        plan.execute(c_in, f_out)
                    else:
                        plan.execute(c_out, f_in)
                    if i >= 2:
                        ms.append(plan.timings()["spread_interp"])
                plan.close()
                rec = {"sweep": name, "type": t, "opts": opts, "ms_median": statistics.median(ms),
                       "ms_min": min(ms), "bins": [info["bin1"], info["bin2"], info["bin3"]][: wl.dim],
                       "msub": info["msub"], "nsub": info["nsub"]}
                print(json.dumps(rec), flush=True)
                key = (name, t)
                if key not in best or rec["ms_median"] < best[key]["ms_median"]:
                    best[key] = rec
        del xs, c_in, f_in, f_out, c_out, flush
        torch.cuda.empty_cache()
    for (name, t), rec in sorted(best.items()):
        print(json.dumps({"sweep_best": name, "type": t, "opts": rec["opts"],
                          "ms_median": rec["ms_median"]}), flush=True)
    return 0


def main():
    args = parse()
    if args.sweep:
        return run_sweep(args)
    wl = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
