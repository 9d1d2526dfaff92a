#!/usr/bin/env python3
"""Benchmark of the streaming log-domain Sinkhorn hot path on GB300.

One step = one pass of the whole hot path over the 50k x 50k, d = 512 point-cloud workload
(X, Y ~ N(0, I/d), uniform weights, eps = 0.1): pack + 100 alternating f/g iterations +
dual loss, the barycentric gradient w.r.t. X, transport application P V and P^T U with
k = 128 columns, and the Hadamard-weighted transport (P .* X Y^T) 1. The headline metric is
Sinkhorn iterations per second (and score evaluations per second); the dominant kernel
(the streaming LSE half-step) is also reported against the measured tensor-core peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--precision bf16|tf32]
  python bench.py --impl reference ...   # the fp64 CPU oracle, bounded sample, host cores

Under torchrun (N > 1) every rank solves its own replica of the problem (the method has
no data-path exchange to shard a single solve across GPUs here); the value is the sum.
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

METRIC = "Sinkhorn iters/sec & score evals/s at n=m=50k vs oracle; % of GB300 roofline"
UNIT = "iters/s"
WORKLOAD_IDX = 3
K_APPLY = 128
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense tensor rates (PFLOP/s): tf32 1.1, bf16 2.25. Used only when no measured tf32
# peak (bench.py --measure-tf32-peak, stored under profiles/) is present.
TF32_OVER_BF16 = 1.1 / 2.25
TF32_PEAK_FILE = os.path.join(ROOT, "profiles", "tf32_peak_gb300.json")
L2_FLUSH_BYTES = 256 << 20
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["flashot", "reference"], default="flashot")
    p.add_argument("--precision", choices=["bf16", "tf32", "tf32x3", "fp32"], default=None,
                   help="contraction precision (default: bf16; fp32 for the d < 32 workloads)")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    p.add_argument("--no-tf32", action="store_true",
                   help="skip the tf32 record of the benchmark line")
    p.add_argument("--measure-tf32-peak", action="store_true",
                   help="time torch.matmul 8192^3 with tf32 allowed (best of 10, and back to "
                        "back for 4 s) and print the record; with --write-peak also store it "
                        "as profiles/tf32_peak_gb300.json, which the roofline lines use")
    p.add_argument("--write-peak", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-passes", type=int, default=0, metavar="P",
                   help="profiling driver: pack once, run P f-updates and P g-updates of the "
                        "workload (no timing, no JSON line) and exit; for ncu captures. With "
                        "--diagnostics, then P plan diagnostics and P transport applications "
                        "(k = 128) at those potentials")
    p.add_argument("--n", type=int, default=None, help="override n = m (profiling driver)")
    p.add_argument("--schedule", choices=["alternating", "symmetric"], default="alternating",
                   help="supplementary lines: iteration schedule of the solves")
    p.add_argument("--divergence", action="store_true",
                   help="supplementary line: debiased Sinkhorn divergence (three solves)")
    p.add_argument("--diagnostics", action="store_true",
                   help="supplementary line: plan diagnostics (primal/dual objectives, "
                        "transport cost, marginal errors) of --workload at its solved "
                        "potentials; three streaming passes per step")
    p.add_argument("--tol", type=float, default=None,
                   help="supplementary line: convergence-driven solve of --workload to this "
                        "L1 marginal error (with --eps, --max-iters, --check-every)")
    p.add_argument("--eps", type=float, default=None, help="override eps (--tol, --drift)")
    p.add_argument("--max-iters", type=int, default=5000)
    p.add_argument("--check-every", type=int, default=10)
    p.add_argument("--drift", action="store_true",
                   help="supplementary line: fp32 GPU vs fp64 oracle drift over a long "
                        "low-eps run (n = m = 1000, d = 2, eps = 0.001, 3000 iterations)")
    p.add_argument("--hvp", action="store_true",
                   help="supplementary line: Hessian-vector product of the OT loss w.r.t. X "
                        "on n = m = 50000 points in Uniform[0,1]^3 (eps = 0.05, CG to 1e-6)")
    p.add_argument("--hvp-sweep", action="store_true",
                   help="supplementary line: HVP accuracy against the dense fp64 "
                        "Moore-Penrose reference for eps = 0.1 .. 0.01 (n = m = 200, d = 3)")
    p.add_argument("--sk", action="store_true",
                   help="supplementary line: batched Sinkhorn-Knopp of 4 x 4 matrices "
                        "(B = 2^24 unless --sk-batch, 20 iterations)")
    p.add_argument("--sk-batch", type=int, default=1 << 24)
    p.add_argument("--sk-n", type=int, default=4)
    p.add_argument("--graph", action="store_true",
                   help="supplementary solve lines: also capture one solve into a CUDA graph "
                        "and time its replays")
    p.add_argument("--workload", type=int, default=WORKLOAD_IDX, choices=[1, 2, 3, 4, 5],
                   help="3 (default) is the benchmark line; 1, 2, 4, 5 print supplementary "
                        "lines for the other point-cloud workloads")
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.steps < 1:
        p.error("--steps must be >= 1")
    return args


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x, world, device):
    """The largest of x over all ranks (the timed region ends when the slowest rank does);
    x itself with one rank. device: where the collective's buffer lives (cuda for NCCL,
    cpu for gloo)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank, ms_max, world):
    """Whole-job throughput of independent replicas: every rank processes units_per_rank
    units, the job takes the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_tf32_peak(peaks, peak_src):
    """Sustained tf32 tensor-core peak (TFLOP/s), the median SM clock (MHz) it was measured
    at, and where it comes from: the measured record under profiles/ when present, else
    the bf16 sustained peak x the nominal tf32/bf16 ratio."""
    if os.path.exists(TF32_PEAK_FILE):
        with open(TF32_PEAK_FILE) as fh:
            rec = json.load(fh)
        return (float(rec["tf32_tflops_sustained"]), rec.get("clocks_sustained", {}).get("sm_mhz"),
                "measured tf32_tflops_sustained (profiles/tf32_peak_gb300.json)")
    bf16_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    return (bf16_sus * TF32_OVER_BF16, peak_clock_mhz(peaks),
            f"{peak_src} bf16_tflops_sustained x 1.1/2.25 (nominal ratio)")


def peak_clock_mhz(peaks):
    """Median SM clock (MHz) under which the sustained bf16 peak was measured, or None."""
    c = peaks.get("clocks_under_load") or {}
    v = c.get("sm_mhz_median")
    return float(v) if v else None


def clock_matched(frac, run_mhz, peak_mhz):
    """The roofline fraction with the peak rescaled from the clock it was measured at to
    the clock this run saw (time x clock is the work per clock)."""
    if not frac or not run_mhz or not peak_mhz:
        return None
    return frac * float(peak_mhz) / float(run_mhz)


def device_sms(dev=0):
    """Streaming multiprocessors of the device (read from the device, not assumed)."""
    import torch
    return int(torch.cuda.get_device_properties(dev).multi_processor_count)


def run_clock_hz(clk, peaks):
    """SM clock for unit-count peaks (FP32 lanes, SFU): the median sampled during the
    timed region, else the maximum clock. Returns (Hz, label)."""
    if clk and clk.get("sm_mhz"):
        return float(clk["sm_mhz"]) * 1e6, "median SM clock sampled during the timed region"
    return float(peaks.get("sm_max_mhz", 2070.0)) * 1e6, "maximum SM clock (no samples)"


def workload_config(prec, accumulate="f32 scores/LSE, f64 loss"):
    return {
        "workload": "pc50k_d512_grad: n=m=50000, d=512, X,Y~N(0,I/d) fp32, uniform weights, "
                    "eps=0.1, 100 alternating iterations + dual loss + grad wrt X + P.V and "
                    "P^T.U (k=128) + Hadamard (P.*XY^T)1",
        "n": 50000, "m": 50000, "d": 512, "iters": 100, "k_apply": K_APPLY,
        "contraction": prec, "accumulate": accumulate,
        "l2": "flushed before every step (256 MiB write inside the timed region); "
              "working set 2x51 MB bf16 operands",
        "seed": 1000 + WORKLOAD_IDX,
    }


# ---------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs (read-only query)."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on a bounded sample of the same workload
# ---------------------------------------------------------------------------------------
def oracle_sample(pr, target_s=10.0):
    """Time the oracle's f-update on a subset of rows of the full workload and extrapolate
    to iterations per second of the whole problem (one iteration = an f-update over n rows
    plus a g-update over m rows, each against the full other cloud)."""
    import numpy as np

    import oracle
    g = np.zeros(pr.m)
    eps = float(pr.eps_schedule[0])
    r = 4 * oracle.num_threads()
    while True:
        rows = np.linspace(0, pr.n - 1, r).astype(np.int64)
        t0 = time.perf_counter()
        oracle.half_step_f(pr.X, pr.Y, pr.b, g, eps, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or r >= pr.n:
            break
        r = int(min(pr.n, max(2 * r, r * 0.8 * target_s / max(dt, 1e-3))))
    per_row = dt / r
    iter_s = per_row * pr.n + per_row * pr.m  # n = m rows of equal cost for the g-update
    return {"value": 1.0 / iter_s, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "rows": int(r),
            "sample": f"f-update of {r} of {pr.n} rows against all {pr.m} columns (d={pr.d}, "
                      f"fp64), {dt:.1f} s; iteration time extrapolated as (n+m) x per-row time"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from workloads import workload
    pr = workload(WORKLOAD_IDX)
    samples = []
    step_s = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        s = oracle_sample(pr, target_s=8.0)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            samples.append(s)
            step_s.append(dt)
    vals = [s["value"] for s in samples]
    v = statistics.median(vals)
    full_step_s = 100.0 / v  # one step of the workload = 100 iterations
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        # what each timed step executed: one bounded row sample of the f-update
        "ms_per_step": statistics.median(step_s) * 1e3,
        "extrapolated": True,
        "sampled_rows_per_step": samples[-1]["rows"],
        "extrapolated_ms_per_full_step": full_step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, same generator as the GPU arm)",
        "config": workload_config("f64", "f64 (CPU oracle, dense loops, no tiling)"),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": samples[-1]["cores"],
                         "kind": "oracle", "sample": samples[-1]["sample"]},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "fp64 plain-loop CPU oracle timed on the host cores. Each timed step runs "
                "the f-update for a bounded sample of rows against all columns "
                "(ms_per_step is that sample's wall time); value is the iterations/s of "
                "the whole 50k x 50k problem extrapolated from it as (n + m) x per-row time",
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------
# The sources that define the tensor-core LSE kernel: its translation unit and the headers
# whose code it runs. (fma_kernels.cuh and flashot.h are included there as well but hold
# nothing the LSE kernel executes: the split reduction of the tf32 weighted sums, and the
# public API.) The recorded ncu traffic is valid while these are unchanged.
LSE_KERNEL_SOURCES = ("tc_kernels.cu", "lse_epilogue.cuh", "common.cuh", "pack_kernels.cuh", "ptx.cuh",
                      "tc_api.h", "tc_host.h", "trace.h")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "log_domain_sinkhorn_gb300", "csrc")
    for name in LSE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(prec):
    """DRAM bytes per launch of the LSE kernel from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "lse_tc_kernel_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    ent = rec.get(prec)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_full_launch")


# Peak fp32 FMA throughput used for the CUDA-core path: SMs (read from the device) x 128
# FP32 lanes x 2 flops per FMA x the SM clock sampled during the timed region. The SFU rate
# for ex2.approx.ftz.f32 is 32 per clock per SM (measured with a throughput probe on GB300:
# 32.7 per clock); the SFU reciprocal rate is 16.
FP32_LANES_PER_SM = 128
SFU_EX2_PER_SM_CLK = 32
SFU_RCP_PER_SM_CLK = 16


def run_other_workload(args):
    """Supplementary measurement of workloads 1, 2, 4 (solves) and 5 (transport application
    at converged potentials): one JSON line each, in that workload's own unit."""
    import torch

    import log_domain_sinkhorn_gb300 as lds
    from workloads import workload
    idx = args.workload
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pr = workload(idx)
    prec = args.precision or ("fp32" if pr.d < 32 else "bf16")
    n, m, d = pr.n, pr.m, pr.d
    X = torch.from_numpy(pr.X).to(dev)
    Y = torch.from_numpy(pr.Y).to(dev)
    a = None if pr.uniform_weights else torch.from_numpy(pr.a).to(dev)
    b = None if pr.uniform_weights else torch.from_numpy(pr.b).to(dev)
    sched = [float(e) for e in pr.eps_schedule]
    k = pr.V.shape[1] if pr.V is not None else 0
    ws = lds.Workspace(lds.workspace_bytes(n, m, d, k, prec))
    f = torch.empty(n, device=dev)
    g = torch.empty(m, device=dev)
    loss = torch.empty((), dtype=torch.float64, device=dev)
    nm = float(n) * float(m)
    if args.diagnostics:
        lds.sinkhorn_solve(X, Y, a, b, sched, pr.iters_per_stage, precision=prec, f_out=f,
                           g_out=g, loss_out=loss, workspace=ws)
        res = torch.empty(6, dtype=torch.float64, device=dev)
        dws = lds.Workspace(int(lds.library().flashot_diagnostics_workspace_bytes(
            n, m, d, lds._flags(prec))))
        eps = sched[-1]

        def step():
            lds.plan_diagnostics(X, Y, f, g, eps, a, b, precision=prec, out=res, workspace=dws,
                                 as_dict=False)
        # r = P 1, c = P^T 1 and the Hadamard sums: three streaming passes over the n x m
        # scores (plus O(n + m) packing and the fp64 reduction)
        units_per_step, unit, scores_per_step = 1, "plan diagnostics/s", 3 * nm
        hot = lds.KernelTimer.WSUM
    elif idx == 5:
        lds.sinkhorn_solve(X, Y, a, b, sched, pr.iters_per_stage, precision=prec, f_out=f,
                           g_out=g, loss_out=loss, workspace=ws)
        V = torch.from_numpy(pr.V).to(dev)
        U = torch.from_numpy(pr.U).to(dev)
        PV = torch.empty((n, k), device=dev)
        PtU = torch.empty((m, k), device=dev)
        h = torch.empty(n, device=dev)
        eps = sched[0]

        def step():
            lds.transport_apply(X, Y, f, g, eps, V, a, b, precision=prec, out=PV, workspace=ws,
                                reuse_pack=True)
            lds.transport_apply(X, Y, f, g, eps, U, a, b, transpose=True, precision=prec,
                                out=PtU, workspace=ws, reuse_pack=True)
            lds.transport_hadamard_xy(X, Y, f, g, eps, a, b, precision=prec, out=h,
                                      workspace=ws, reuse_pack=True)
        units_per_step, unit, scores_per_step = 3, "transport applications/s", 3 * nm
        hot = lds.KernelTimer.WSUM
    elif args.divergence:
        res = torch.empty(4, dtype=torch.float64, device=dev)
        dws = lds.Workspace(int(lds.library().flashot_divergence_workspace_bytes(
            n, m, d, lds._flags(prec, schedule=args.schedule))))

        def step():
            lds.sinkhorn_divergence(X, Y, a, b, sched, pr.iters_per_stage, precision=prec,
                                    schedule=args.schedule, out=res, workspace=dws)
        units_per_step, unit = 1, "divergences/s"
        # Scores evaluated: the X-Y solve runs two passes per iteration; with the symmetric
        # schedule the self-transport solves (X-X, Y-Y) run one (f == g throughout).
        self_passes = 1 if args.schedule == "symmetric" else 2
        scores_per_step = (2 * n * m + self_passes * (n * n + m * m)) * pr.total_iters
        hot = lds.KernelTimer.LSE
    else:
        def step():
            lds.sinkhorn_solve(X, Y, a, b, sched, pr.iters_per_stage, precision=prec, f_out=f,
                               g_out=g, loss_out=loss, workspace=ws, schedule=args.schedule)
        units_per_step, unit = pr.total_iters, "iters/s"
        scores_per_step = 2 * nm * pr.total_iters
        hot = lds.KernelTimer.LSE
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    # Throughput: the steps alone. The per-launch event timer records an event between
    # every two kernels, which serialises programmatically dependent launches, so it runs
    # in a second loop over the same steps, for the hot kernel's average duration.
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    launches0 = lds.launch_count()
    clocks = ClockSampler(0).start()
    time.sleep(0.3)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk_rec = clocks.stop()
    ms = e0.elapsed_time(e1)
    launches = lds.launch_count() - launches0
    timer = lds.KernelTimer(cap=args.steps * 2200).start()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    n_hot, ms_hot = timer.read(hot)
    timer.stop()
    if lds.workspace_status(ws) != 0:
        raise RuntimeError("device timeout reported")
    peaks, peak_src = load_peaks()
    sms = device_sms()
    clk, clk_src = run_clock_hz(clk_rec, peaks)
    avg = ms_hot / max(n_hot, 1) / 1e3
    # Scores per timed launch of the hot kernel class: the streaming solve launches one LSE
    # pass per half-step; the single-launch solves (the cluster solve of small fp32
    # problems, the persistent solve of short tensor-core contractions) cover the whole
    # solve.
    per_launch_scores = scores_per_step * args.steps / max(n_hot, 1)
    if prec == "fp32":
        roof = {"bound": "alu", "achieved": 2.0 * d * per_launch_scores / avg / 1e12,
                "peak": sms * FP32_LANES_PER_SM * 2 * clk / 1e12, "unit": "TFLOP/s (fp32 FMA)",
                "peak_source": f"{sms} SMs x 128 FP32 lanes x 2 x {clk_src}"}
    else:
        bf16_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        tf32, tf32_mhz, tf32_src = load_tf32_peak(peaks, peak_src)
        # Algorithmic flops (2d per score); split tf32 runs three tf32 contractions, so its
        # ceiling for the algorithmic rate is a third of the tf32 peak.
        roof = {"bound": "tensor", "achieved": 2.0 * d * per_launch_scores / avg / 1e12,
                "peak": bf16_sus if prec == "bf16" else (tf32 / 3 if prec == "tf32x3" else tf32),
                "unit": "TFLOP/s",
                "peak_source": (f"{peak_src} bf16_tflops_sustained" if prec == "bf16" else
                                tf32_src + (" / 3 (split tf32)" if prec == "tf32x3" else ""))}
        pk_mhz = peak_clock_mhz(peaks) if prec == "bf16" else tf32_mhz
        roof["frac_clock_matched"] = clock_matched(roof["achieved"] / roof["peak"],
                                                   clk_rec.get("sm_mhz"), pk_mhz)
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["sfu_frac"] = (per_launch_scores / avg) / (sms * SFU_EX2_PER_SM_CLK * clk)
    # The governing roofline is the unit whose floor for this work is longest, i.e. the
    # larger of the two fractions at the run's clock (tensor or FMA pipe, the tensor peak
    # rescaled to the run clock, against the SFU's one ex2 per score).
    own = roof.get("frac_clock_matched") or roof["frac"]
    roof["governing"] = "sfu (ex2)" if roof["sfu_frac"] > own else roof["bound"]
    roof["governing_frac"] = max(roof["sfu_frac"], own)
    if prec == "fp32" and d <= 32:
        # FMA-pipe work per score of the small-d CUDA-core LSE: the padded dot product
        # (d_pad lanes), kappa * dot + bias, the max shift and the sum (the max itself runs
        # on the ALU pipe): d_pad + 3 lane operations against 128 lanes per SM per clock.
        d_pad = (d + 3) // 4 * 4
        roof["fma_pipe_frac"] = ((per_launch_scores / avg) * (d_pad + 3)
                                 / (sms * FP32_LANES_PER_SM * clk))
    roof["avg_launch_ms"] = avg * 1e3
    roof["launches_timed"] = n_hot
    roof["scores_per_launch"] = per_launch_scores
    graph = None
    if args.graph and idx != 5 and not args.divergence and not args.diagnostics:
        # The same solve captured once into a CUDA graph (torch's capture stream is the
        # current stream the binding passes) and replayed: no per-launch host work.
        cg = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()  # the first call on a stream may set kernel attributes; keep it out
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        l0 = lds.launch_count()
        with torch.cuda.graph(cg):
            step()
        per_solve_launches = lds.launch_count() - l0
        for _ in range(args.warmup):
            cg.replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(args.steps):
            cg.replay()
        g1.record()
        torch.cuda.synchronize()
        gms = g0.elapsed_time(g1)
        graph = {"value": units_per_step * args.steps / (gms / 1e3), "unit": unit,
                 "ms_per_step": gms / args.steps, "kernels_per_replay": int(per_solve_launches),
                 "speedup_vs_direct": ms / gms}
    line = {"metric": f"workload {idx} ({pr.name}) throughput"
                      + (" [debiased divergence]" if args.divergence else "")
                      + (" [plan diagnostics]" if args.diagnostics else "")
                      + (" [symmetric schedule]" if args.schedule == "symmetric" else ""),
            "supplementary": True,
            "value": units_per_step * args.steps / (ms / 1e3), "unit": unit,
            "score_evals_per_s": scores_per_step * args.steps / (ms / 1e3),
            "ms_per_step": ms / args.steps, "steps": args.steps, "warmup": args.warmup,
            "dtype": prec, "config": {"workload": pr.name, "n": n, "m": m, "d": d,
                                      "eps": sched if len(sched) > 1 else sched[0],
                                      "iters_per_stage": pr.iters_per_stage},
            "roofline": roof, "clocks": clk_rec, "gpu_launches": int(launches)}
    if graph is not None:
        line["cuda_graph"] = graph
    if args.diagnostics:
        if lds.workspace_status(dws) != 0:
            raise RuntimeError("device timeout reported")
        line["diagnostics"] = dict(zip(("primal", "dual", "transport_cost", "row_err",
                                        "col_err", "mass"), res.cpu().tolist()))
    print(json.dumps(line), flush=True)


def _problem_on_device(pr, dev):
    import torch
    X = torch.from_numpy(pr.X).to(dev)
    Y = torch.from_numpy(pr.Y).to(dev)
    a = None if pr.uniform_weights else torch.from_numpy(pr.a).to(dev)
    b = None if pr.uniform_weights else torch.from_numpy(pr.b).to(dev)
    return X, Y, a, b


def run_convergence(args):
    """Supplementary line: the convergence-driven solve (stop when the L1 row-marginal error
    measured inside the f-update falls below --tol) on a workload at one eps. Reports the
    iterations and time to tolerance, and the cost of the checks against a fixed-iteration
    solve of the same length."""
    import torch

    import log_domain_sinkhorn_gb300 as lds
    from workloads import workload
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pr = workload(args.workload)
    prec = args.precision or ("fp32" if pr.d < 32 else "bf16")
    eps = float(args.eps if args.eps is not None else pr.eps_schedule[-1])
    n, m, d = pr.n, pr.m, pr.d
    X, Y, a, b = _problem_on_device(pr, dev)
    ws = lds.Workspace(lds.workspace_bytes(n, m, d, 0, prec))
    f = torch.empty(n, device=dev)
    g = torch.empty(m, device=dev)
    loss = torch.empty((), dtype=torch.float64, device=dev)
    res = {}

    def tol_solve():
        res["out"] = lds.sinkhorn_solve_tol(X, Y, a, b, eps, args.tol, args.max_iters,
                                            args.check_every, precision=prec, f_out=f,
                                            g_out=g, loss_out=loss, workspace=ws)

    for _ in range(args.warmup):
        tol_solve()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        tol_solve()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    _, _, _, iters, err, hist = res["out"]
    ms_tol = statistics.median(times)
    # the same number of iterations without checks
    fixed = []
    for i in range(args.warmup + args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        lds.sinkhorn_solve(X, Y, a, b, eps, iters, precision=prec, f_out=f, g_out=g,
                           loss_out=loss, workspace=ws)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            fixed.append(e0.elapsed_time(e1))
    ms_fixed = statistics.median(fixed)
    if lds.workspace_status(ws) != 0:
        raise RuntimeError("device timeout reported")
    line = {"metric": f"workload {args.workload} ({pr.name}) convergence-driven solve",
            "supplementary": True, "value": iters / (ms_tol / 1e3), "unit": "iters/s",
            "ms_to_tolerance": ms_tol, "iters_to_tolerance": iters, "final_l1_error": err,
            "reached": bool(0 <= err < args.tol),
            "errors_at_checks": [h for h in hist[:: max(1, len(hist) // 20)]],
            "ms_fixed_same_iters": ms_fixed,
            "check_overhead_frac": (ms_tol - ms_fixed) / ms_fixed,
            "steps": args.steps, "warmup": args.warmup, "dtype": prec,
            "config": {"workload": pr.name, "n": n, "m": m, "d": d, "eps": eps,
                       "tol": args.tol, "max_iters": args.max_iters,
                       "check_every": args.check_every, "start": "g = 0"}}
    print(json.dumps(line), flush=True)


def run_drift(args):
    """Supplementary line: drift of the fp32 GPU iterates from the fp64 oracle over a long
    low-eps run (Uniform[0,1]^2 clouds, n = m = 1000, eps = 0.001, 3000 iterations; the
    L1 marginal error falls about 10x per 450 iterations). Reports the potentials' error
    as given and after removing the constant shift (f + c, g - c) that leaves the plan
    unchanged, the loss error, and the measured marginal errors of both runs."""
    import numpy as np
    import torch

    import log_domain_sinkhorn_gb300 as lds
    import oracle
    from workloads import make_problem
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    n, d, eps = 1000, 2, float(args.eps if args.eps is not None else 0.001)
    iters, c = min(args.max_iters, 3000), 100
    pr = make_problem(n, n, d, x_dist="unif01", weights="uniform", seed=4242)
    X, Y, a, b = _problem_on_device(pr, dev)
    out = {}
    for prec in ([args.precision] if args.precision else ["fp32", "tf32x3"]):
        f, g, loss, done, err, hist = lds.sinkhorn_solve_tol(X, Y, a, b, eps, 0.0, iters, c,
                                                             precision=prec)
        out[prec] = (f.cpu().numpy().astype(np.float64), g.cpu().numpy().astype(np.float64),
                     float(loss.cpu()), np.asarray(hist))
    t0 = time.perf_counter()
    f_r, g_r, loss_r, _, _, hist_r = oracle.solve_tol(pr.X, pr.Y, pr.a, pr.b, eps, 0.0, iters,
                                                      c, history=True)
    t_oracle = time.perf_counter() - t0
    scale = max(np.abs(f_r).max(), np.abs(g_r).max())
    res = {}
    for prec, (f, g, loss, hist) in out.items():
        shift = (np.mean(f - f_r) - np.mean(g - g_r)) / 2.0
        res[prec] = {
            "pot_err_raw": float(max(np.abs(f - f_r).max(), np.abs(g - g_r).max()) / scale),
            "pot_err_shift_removed": float(max(np.abs(f - shift - f_r).max(),
                                               np.abs(g + shift - g_r).max()) / scale),
            "constant_shift": float(shift),
            "loss_rel_err": abs(loss - loss_r) / abs(loss_r),
            "l1_error_at_checks": [float(x) for x in hist[4::5]],
        }
    line = {"metric": "fp32 vs fp64 drift, low-eps long run", "supplementary": True,
            "value": max(r["pot_err_raw"] for r in res.values()),
            "unit": "relative L-inf potential error after the run (max over precisions)",
            "results": res, "oracle_l1_error_at_checks": [float(x) for x in hist_r[4::5]],
            "fp32_resolution_of_l1_error": 4.0 * float(np.spacing(np.float32(scale))) / eps,
            "oracle_seconds": t_oracle, "oracle_cores": oracle.num_threads(),
            "config": {"workload": "unif01 2-D clouds, n=m=1000, uniform weights", "eps": eps,
                       "iters": iters, "check_every": c, "seed": 4242}}
    print(json.dumps(line), flush=True)


def run_hvp(args):
    """Supplementary line: the streaming Hessian-vector product (fp32 CUDA-core passes, CG
    Schur solve to a relative residual of 1e-6) on n = m = 50000 points in Uniform[0,1]^3,
    uniform weights, eps = 0.05, at potentials from a convergence-driven solve (L1 marginal
    error < 1e-5), V ~ N(0, 1). One step = one H V."""
    import numpy as np
    import torch

    import log_domain_sinkhorn_gb300 as lds
    from workloads import make_problem
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    n = args.n or 50000
    d, eps = 3, float(args.eps if args.eps is not None else 0.05)
    pr = make_problem(n, n, d, x_dist="unif01", weights="uniform", seed=5150)
    X, Y, a, b = _problem_on_device(pr, dev)
    V = torch.from_numpy(np.random.default_rng(5151).normal(size=(n, d)).astype(np.float32)).to(dev)
    f, g, _, iters_solve, err, _ = lds.sinkhorn_solve_tol(X, Y, a, b, eps, 1e-5, 5000, 10,
                                                          precision="fp32")
    ws = lds.Workspace(int(lds.library().flashot_hvp_workspace_bytes(n, n, d, 1)))
    out = torch.empty((n, d), device=dev)
    res = {}

    def step():
        res["r"] = lds.ot_hvp_x(X, Y, f, g, eps, V, a, b, cg_tol=1e-6, out=out, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    timer = lds.KernelTimer(cap=args.steps * 4000).start()
    launches0 = lds.launch_count()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(0).start()
    time.sleep(0.3)
    times = []
    for _ in range(args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    launches = lds.launch_count() - launches0
    clk_rec = clocks.stop()
    n_ws, ms_ws = timer.read(lds.KernelTimer.WSUM)
    n_ot, ms_ot = timer.read(lds.KernelTimer.OTHER)
    timer.stop()
    if lds.workspace_status(ws) != 0:
        raise RuntimeError("device timeout reported")
    _, cg_iters, rel = res["r"]
    ms = statistics.median(times)
    peaks, _ = load_peaks()
    sms = device_sms()
    clk, clk_src = run_clock_hz(clk_rec, peaks)
    nm = float(n) * float(n)
    passes = 2 * cg_iters + 5  # CG: P p and P^T t; plus [PY|r], [P^T V|P^T s|c], T, rhs, final
    pass_avg = ms_ws / max(n_ws, 1) / 1e3
    # FMA-pipe lane operations per score of each streaming pass (d = 3, padded to 4): the
    # exponent (4: kappa rides on the row coordinates, the dot starts from c_j and the
    # padding lane carries the row bias r_i), then the weighted sums at the kernel's padded
    # output width: 1 for P t / P^T t (1 + 2 per CG iteration), 4 for [PY | r] and
    # [P diag(z) Y | P z], 8 for [P^T V | P^T s | c] (5 columns), and 4 for the curvature
    # pass T plus its dot <u_i, y_j> (4) and the product with the weight (1). The ex2 (one
    # per score) runs on the SFU at 32 per clock per SM, never the limit here.
    d_pad = 4
    lane_ops = nm * ((d_pad + 1) * (1 + 2 * cg_iters) + (d_pad + 4) * 2 + (d_pad + 8)
                     + (d_pad + 4 + d_pad + 1))
    passes_s = ms_ws / args.steps / 1e3
    line = {"metric": "Hessian-vector products of the OT loss w.r.t. X", "supplementary": True,
            "value": 1e3 / ms, "unit": "HVPs/s", "ms_per_hvp": ms, "cg_iterations": cg_iters,
            "cg_rel_residual": rel, "streaming_passes_per_hvp": passes,
            "ms_per_cg_iteration": ms / max(cg_iters, 1),
            "kernels_ms_per_hvp": {"streaming_passes": ms_ws / args.steps,
                                   "other": ms_ot / args.steps},
            "roofline": {"bound": "alu (fp32 FMA pipe)",
                         "kernel": "wsum_fma_pair (streaming passes)",
                         "achieved": lane_ops / passes_s / 1e12,
                         "peak": sms * FP32_LANES_PER_SM * clk / 1e12,
                         "unit": "T FMA-pipe lane-ops/s",
                         "peak_source": f"{sms} SMs x 128 FP32 lanes x {clk_src}",
                         "lane_ops_per_hvp": lane_ops,
                         "sfu_frac": (nm / pass_avg) / (sms * SFU_EX2_PER_SM_CLK * clk),
                         "avg_pass_ms": pass_avg * 1e3},
            "clocks": clk_rec,
            "steps": args.steps, "warmup": args.warmup, "dtype": "fp32",
            "gpu_launches": int(launches),
            "config": {"workload": "hvp50k_d3: n=m=%d, d=3, Uniform[0,1]^3, uniform weights" % n,
                       "eps": eps, "potentials": f"solve to L1 marginal error {err:.2e} "
                                                 f"({iters_solve} iterations)",
                       "V": "N(0,1), seed 5151", "cg_tol": 1e-6}}
    line["roofline"]["frac"] = line["roofline"]["achieved"] / line["roofline"]["peak"]
    print(json.dumps(line), flush=True)


def run_hvp_sweep(args):
    """Supplementary line: relative L2 error of the streaming HVP against the dense fp64
    Moore-Penrose reference, and CG iterations, for eps = 0.1, 0.05, 0.02, 0.01 (n = m = 200
    points in Uniform[0,1]^3, uniform weights, potentials converged by the oracle and cast to
    fp32, V ~ N(0, 1), CG to a relative residual of 1e-6)."""
    import numpy as np
    import torch

    import log_domain_sinkhorn_gb300 as lds
    import oracle
    from workloads import make_problem
    torch.cuda.set_device(0)
    n, d = 200, 3
    pr = make_problem(n, n, d, x_dist="unif01", weights="uniform", seed=6060)
    V = np.random.default_rng(6061).normal(size=(n, d)).astype(np.float32)
    dv = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    rows = []
    for eps in (0.1, 0.05, 0.02, 0.01):
        f, g, _, it, err = oracle.solve_tol(pr.X, pr.Y, pr.a, pr.b, eps, 1e-12, 400000, 10)
        f32, g32 = f.astype(np.float32), g.astype(np.float32)
        ref = oracle.hvp_x(pr.X, pr.Y, pr.a, pr.b, f32, g32, eps, V)
        HV, cg_it, rel = lds.ot_hvp_x(dv(pr.X), dv(pr.Y), dv(f32), dv(g32), eps, dv(V),
                                      dv(pr.a), dv(pr.b), cg_tol=1e-6)
        e = float(np.linalg.norm(HV.cpu().numpy() - ref) / np.linalg.norm(ref))
        rows.append({"eps": eps, "rel_l2_error": e, "cg_iterations": cg_it,
                     "cg_rel_residual": rel, "oracle_solve_iterations": it})
    line = {"metric": "HVP accuracy vs dense Moore-Penrose reference", "supplementary": True,
            "value": max(r["rel_l2_error"] for r in rows),
            "unit": "max relative L2 error over eps", "results": rows, "dtype": "fp32",
            "config": {"workload": "n=m=200, d=3, Uniform[0,1]^3, uniform weights",
                       "V": "N(0,1), seed 6061", "cg_tol": 1e-6}}
    print(json.dumps(line), flush=True)


def run_sk(args):
    """Supplementary line: batched Sinkhorn-Knopp projection of B tiny n x n matrices (the
    mHC setting of "Fused & Furious": n = 4, 20 iterations, B up to 2^24), logits ~ N(0, 1).
    Algorithmic bytes: the logits read and P written, 2 B n^2 4 bytes. Inputs larger than
    L2 at the default B (1.07 GB each way); smaller batches flush L2 between steps."""
    import numpy as np
    import torch

    import log_domain_sinkhorn_gb300 as lds
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    B, n, n_iter = args.sk_batch, args.sk_n, 20
    g = torch.Generator(device=dev).manual_seed(4444)
    H = torch.randn((B, n, n), device=dev, generator=g)
    P = torch.empty_like(H)
    bytes_step = 2.0 * B * n * n * 4
    flush = None if bytes_step > 4 * L2_FLUSH_BYTES else torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        lds.sinkhorn_knopp_batched(H, n_iter, out=P)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(0).start()
    times = []
    for _ in range(args.steps):
        if flush is not None:
            flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        lds.sinkhorn_knopp_batched(H, n_iter, out=P)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    clk = clocks.stop()
    ms = statistics.median(times)
    peaks, src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        Bs = min(B, 1 << 20)
        Hs = H[:Bs].cpu().numpy()
        t0 = time.perf_counter()
        oracle.sinkhorn_knopp(Hs, n_iter)
        dt = time.perf_counter() - t0
        cpu = {"value": Bs / dt, "unit": "matrices/s", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": f"the first {Bs} matrices, {dt:.2f} s"}
    # Roofline: the algorithm as stated needs per matrix 2 n^2 n_iter + 2 n^2 FMA-pipe ops
    # (row and column sums, the final scaling), n^2 + 2 n n_iter SFU ops (exp and one
    # reciprocal per sum) and 2 n^2 4 bytes of HBM traffic. Its time floor is the largest of
    # the three at FP32 = 128 lanes, SFU reciprocal = 16 lanes per clock per SM.
    sms = device_sms()
    clk_hz, clk_src = run_clock_hz(clk, peaks)
    fma_ops = 2 * n * n * n_iter + 2 * n * n
    xu_ops = n * n + 2 * n * n_iter
    t_fma = B * fma_ops / (sms * FP32_LANES_PER_SM * clk_hz)
    t_xu = B * xu_ops / (sms * SFU_RCP_PER_SM_CLK * clk_hz)
    t_hbm = bytes_step / (hbm * 1e9)
    t_floor = max(t_fma, t_xu, t_hbm)
    line = {"metric": "batched Sinkhorn-Knopp (mHC %dx%d, %d iterations)" % (n, n, n_iter),
            "supplementary": True, "value": B / (ms / 1e3), "unit": "matrices/s",
            "ms_per_step": ms, "ms_q01_q99": [float(np.quantile(times, 0.01)),
                                               float(np.quantile(times, 0.99))],
            "steps": args.steps, "warmup": args.warmup, "dtype": "fp32",
            "roofline": {"bound": "alu", "achieved": B / (ms / 1e3), "peak": B / t_floor,
                         "unit": "matrices/s", "frac": t_floor / (ms / 1e3),
                         "floor_ms": {"fma_pipe": t_fma * 1e3, "sfu": t_xu * 1e3,
                                      "hbm": t_hbm * 1e3},
                         "per_matrix": {"fma_ops": fma_ops, "sfu_ops": xu_ops,
                                        "bytes": 2 * n * n * 4},
                         "hbm_achieved_gbs": bytes_step / (ms / 1e3) / 1e9,
                         "hbm_frac": bytes_step / (ms / 1e3) / 1e9 / hbm,
                         "peak_source": f"{src} hbm_gbs; FP32 and SFU from unit counts x "
                                        f"{sms} SMs x {clk_src}"},
            "clocks": clk, "cpu_baseline": cpu, "gpu_launches": args.steps,
            "config": {"workload": "B=%d matrices %dx%d, logits N(0,1), %d iterations" % (B, n, n, n_iter),
                       "l2": "inputs larger than L2" if flush is None else "L2 flushed before each step"}}
    print(json.dumps(line), flush=True)


def run_gpu(args):
    import numpy as np
    import torch

    import log_domain_sinkhorn_gb300 as lds
    from workloads import workload

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    prec = args.precision

    pr = workload(WORKLOAD_IDX)
    n, m, d = pr.n, pr.m, pr.d
    eps = float(pr.eps_schedule[0])
    iters = pr.iters_per_stage
    X = torch.from_numpy(pr.X).to(dev)
    Y = torch.from_numpy(pr.Y).to(dev)
    V = torch.from_numpy(pr.V).to(dev)
    U = torch.from_numpy(pr.U).to(dev)
    ws = lds.Workspace(lds.workspace_bytes(n, m, d, K_APPLY, prec))
    f = torch.empty(n, device=dev)
    g = torch.empty(m, device=dev)
    loss = torch.empty((), dtype=torch.float64, device=dev)
    grad = torch.empty((n, d), device=dev)
    PV = torch.empty((n, K_APPLY), device=dev)
    PtU = torch.empty((m, K_APPLY), device=dev)
    h = torch.empty(n, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(Xs, Ys, Vs, Us):
        flush.zero_()
        lds.sinkhorn_solve(Xs, Ys, None, None, eps, iters, precision=prec, f_out=f, g_out=g,
                           loss_out=loss, workspace=ws)
        lds.ot_grad_x(Xs, Ys, g, eps, precision=prec, out=grad, workspace=ws, reuse_pack=True)
        lds.transport_apply(Xs, Ys, f, g, eps, Vs, precision=prec, out=PV, workspace=ws,
                            reuse_pack=True)
        lds.transport_apply(Xs, Ys, f, g, eps, Us, transpose=True, precision=prec, out=PtU,
                            workspace=ws, reuse_pack=True)
        lds.transport_hadamard_xy(Xs, Ys, f, g, eps, precision=prec, out=h, workspace=ws,
                                  reuse_pack=True)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step(X, Y, V, U)
    torch.cuda.synchronize()
    if lds.workspace_status(ws) != 0:
        raise RuntimeError("a kernel reported a device timeout during warm-up")

    # ---- timed region: inputs resident in HBM --------------------------------------------
    timer = lds.KernelTimer(cap=args.steps * 600).start()
    clocks = ClockSampler(local).start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    launches0 = lds.launch_count()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    e0.record(stream)
    marks[0].record(stream)
    for i in range(args.steps):
        step(X, Y, V, U)
        marks[i + 1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    launches = lds.launch_count() - launches0
    per_step = [marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    n_lse, ms_lse = timer.read(lds.KernelTimer.LSE)
    n_ws, ms_ws = timer.read(lds.KernelTimer.WSUM)
    n_ot, ms_ot = timer.read(lds.KernelTimer.OTHER)
    timer.stop()
    if lds.workspace_status(ws) != 0:
        raise RuntimeError("a kernel reported a device timeout in the timed region")

    total_iters = args.steps * iters * world
    value = replica_throughput(args.steps * iters, ms, world)
    nm = float(n) * float(m)
    scores_per_step = (2 * iters + 5) * nm  # solve + grad (2 passes) + 2 applies + Hadamard
    score_evals = scores_per_step * args.steps * world / (ms / 1e3)

    peaks, peak_src = load_peaks()
    bf16_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    tf32_sus, tf32_mhz, tf32_src = load_tf32_peak(peaks, peak_src)

    def lse_peak(p):
        # Split tf32 runs three tf32 contractions per algorithmic one: its ceiling for the
        # algorithmic rate is a third of the tf32 peak.
        if p == "bf16":
            return bf16_sus, peak_clock_mhz(peaks), f"{peak_src} bf16_tflops_sustained"
        div = 3 if p == "tf32x3" else 1
        return (tf32_sus / div, tf32_mhz,
                tf32_src + (" / 3 (split tf32)" if p == "tf32x3" else ""))

    peak, peak_mhz, peak_label = lse_peak(prec)
    lse_avg_ms = ms_lse / max(n_lse, 1)
    flops_per_launch = 2.0 * nm * d
    achieved = flops_per_launch / (lse_avg_ms / 1e3) / 1e12
    traffic = profiled_traffic(prec)

    # ---- the same step with a tf32 contraction (the pages' own precision) ----------------
    tf32_rec = None
    if prec == "bf16" and not args.no_tf32:
        ws32 = lds.Workspace(lds.workspace_bytes(n, m, d, K_APPLY, "tf32"))

        def step32():
            flush.zero_()
            lds.sinkhorn_solve(X, Y, None, None, eps, iters, precision="tf32", f_out=f,
                               g_out=g, loss_out=loss, workspace=ws32)
            lds.ot_grad_x(X, Y, g, eps, precision="tf32", out=grad, workspace=ws32,
                          reuse_pack=True)
            lds.transport_apply(X, Y, f, g, eps, V, precision="tf32", out=PV, workspace=ws32,
                                reuse_pack=True)
            lds.transport_apply(X, Y, f, g, eps, U, transpose=True, precision="tf32",
                                out=PtU, workspace=ws32, reuse_pack=True)
            lds.transport_hadamard_xy(X, Y, f, g, eps, precision="tf32", out=h,
                                      workspace=ws32, reuse_pack=True)

        for _ in range(args.warmup):
            step32()
        torch.cuda.synchronize()
        timer32 = lds.KernelTimer(cap=args.steps * 600).start()
        clocks32 = ClockSampler(local).start()
        time.sleep(0.3)
        barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step32()
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        clk32 = clocks32.stop()
        ms32 = max_over_ranks(t0.elapsed_time(t1), world, dev)
        n32, ms_lse32 = timer32.read(lds.KernelTimer.LSE)
        timer32.stop()
        if lds.workspace_status(ws32) != 0:
            raise RuntimeError("a kernel reported a device timeout in the tf32 region")
        avg32 = ms_lse32 / max(n32, 1)
        ach32 = flops_per_launch / (avg32 / 1e3) / 1e12
        pk32, pk32_mhz, pk32_label = lse_peak("tf32")
        tf32_rec = {
            "value": replica_throughput(args.steps * iters, ms32, world), "unit": UNIT,
            "ms_per_step": ms32 / args.steps, "dtype": "tf32",
            "score_evals_per_s": scores_per_step * args.steps * world / (ms32 / 1e3),
            "roofline": {"bound": "tensor", "achieved": ach32, "peak": pk32,
                         "unit": "TFLOP/s", "frac": ach32 / pk32,
                         "traffic": profiled_traffic("tf32"),
                         "frac_clock_matched": clock_matched(ach32 / pk32, clk32.get("sm_mhz"),
                                                             pk32_mhz),
                         "peak_clock_mhz": pk32_mhz, "avg_launch_ms": avg32,
                         "launches_timed": n32, "peak_source": pk32_label},
            "clocks": clk32,
            "note": "the same step (solve, gradient, both applications, Hadamard) with every "
                    "contraction on tf32 tensor cores, timed after the bf16 region",
        }
        del ws32

    # ---- end to end through the public API with host buffers -----------------------------
    e2e = None
    if not args.no_e2e:
        hX = torch.from_numpy(pr.X).pin_memory()
        hY = torch.from_numpy(pr.Y).pin_memory()
        hV = torch.from_numpy(pr.V).pin_memory()
        hU = torch.from_numpy(pr.U).pin_memory()
        dX, dY, dV, dU = (torch.empty_like(t, device=dev) for t in (hX, hY, hV, hU))
        outs_d = (f, g, loss, grad, PV, PtU, h)
        outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs_d]
        h2d = sum(t.numel() * t.element_size() for t in (hX, hY, hV, hU))
        d2h = sum(t.numel() * t.element_size() for t in outs_d)

        side = torch.cuda.Stream(device=dev)

        def e2e_step():
            # X and Y first, on the compute stream (the solve packs them). V and U go up on
            # a second stream while the solve runs; each result is read back on that stream
            # as soon as the pass that writes it is done. The step ends when every copy has.
            main = torch.cuda.current_stream()
            dX.copy_(hX, non_blocking=True)
            dY.copy_(hY, non_blocking=True)
            side.wait_stream(main)  # the previous step's reads of dV / dU are done
            with torch.cuda.stream(side):
                dV.copy_(hV, non_blocking=True)
                dU.copy_(hU, non_blocking=True)
            vu_ready = side.record_event()
            flush.zero_()
            lds.sinkhorn_solve(dX, dY, None, None, eps, iters, precision=prec, f_out=f,
                               g_out=g, loss_out=loss, workspace=ws)
            solved = main.record_event()
            lds.ot_grad_x(dX, dY, g, eps, precision=prec, out=grad, workspace=ws,
                          reuse_pack=True)
            grad_done = main.record_event()
            main.wait_event(vu_ready)
            lds.transport_apply(dX, dY, f, g, eps, dV, precision=prec, out=PV, workspace=ws,
                                reuse_pack=True)
            pv_done = main.record_event()
            lds.transport_apply(dX, dY, f, g, eps, dU, transpose=True, precision=prec,
                                out=PtU, workspace=ws, reuse_pack=True)
            lds.transport_hadamard_xy(dX, dY, f, g, eps, precision=prec, out=h, workspace=ws,
                                      reuse_pack=True)
            last_done = main.record_event()
            with torch.cuda.stream(side):
                for ev, idx in ((solved, (0, 1, 2)), (grad_done, (3,)), (pv_done, (4,)),
                                (last_done, (5, 6))):
                    side.wait_event(ev)
                    for i in idx:
                        outs_h[i].copy_(outs_d[i], non_blocking=True)
            main.wait_stream(side)

        e2e_step()
        torch.cuda.synchronize()
        barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_e2e = max_over_ranks(t0.elapsed_time(t1), world, dev)
        e2e = {"value": total_iters / (ms_e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e / args.steps,
               "note": "every step: pinned host -> device copy of X, Y, V, U, the step, "
                       "device -> host copy of f, g, loss, grad, P.V, P^T.U, h, all inside "
                       "the timed region; V, U and the read-backs run on a second stream, "
                       "overlapped with the passes that do not need them"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(pr)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "ms_per_step_median": float(np.median(per_step)),
            "ms_per_step_q01_q99": [float(np.quantile(per_step, 0.01)),
                                    float(np.quantile(per_step, 0.99))],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": prec, "data": "synthetic (seeded numpy PCG64, N(0,I/d) point clouds)",
            "config": workload_config(prec),
            "score_evals_per_s": score_evals,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "frac_clock_matched": clock_matched(achieved / peak, clk.get("sm_mhz"),
                                                             peak_mhz),
                         "peak_clock_mhz": peak_mhz, "traffic": traffic,
                         "kernel": "lse_pair_kernel (streaming LSE half-step on 2-SM CTA pairs)",
                         "algorithmic_flops_per_launch": flops_per_launch,
                         "avg_launch_ms": lse_avg_ms, "launches_timed": n_lse,
                         "peak_source": peak_label},
            "kernels_ms_per_step": {"lse": ms_lse / args.steps, "wsum": ms_ws / args.steps,
                                    "other": ms_ot / args.steps,
                                    "launches_per_step": {"lse": n_lse / args.steps,
                                                          "wsum": n_ws / args.steps,
                                                          "other": n_ot / args.steps}},
            "clocks": clk,
            "e2e": e2e,
            "tf32": tf32_rec,
            "gpu_launches": int(launches),
            "cpu_baseline": cpu,
            "replicas": "one independent problem per rank" if world > 1 else None,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_driver(args):
    """A short, self-contained sequence of the hot kernel for profilers: one pack, then
    alternating f- and g-updates of --workload (default: the 50k benchmark workload;
    optionally with n = m overridden)."""
    import torch

    import log_domain_sinkhorn_gb300 as lds
    from workloads import make_problem, WORKLOADS
    spec = dict(WORKLOADS[args.workload])
    if args.n:
        spec["n"] = spec["m"] = args.n
    spec.pop("k", None)
    pr = make_problem(seed=1000 + args.workload, **spec)
    X = torch.from_numpy(pr.X).cuda()
    Y = torch.from_numpy(pr.Y).cuda()
    eps = float(pr.eps_schedule[0])
    ws = lds.Workspace(lds.workspace_bytes(pr.n, pr.m, pr.d, 0, args.precision))
    g = torch.zeros(pr.m, device="cuda")
    f = torch.empty(pr.n, device="cuda")
    lds.sinkhorn_step_f(X, Y, g, eps, precision=args.precision, out=f, workspace=ws)
    for _ in range(args.profile_passes):
        lds.sinkhorn_step_g(X, Y, f, eps, precision=args.precision, out=g, workspace=ws,
                            reuse_pack=True)
        lds.sinkhorn_step_f(X, Y, g, eps, precision=args.precision, out=f, workspace=ws,
                            reuse_pack=True)
    extra = ""
    if args.diagnostics:
        # then the weighted-sum passes at those potentials: per round one plan diagnostics
        # (P 1, P^T 1, Hadamard) and one P V with k = 128
        dws = lds.Workspace(int(lds.library().flashot_diagnostics_workspace_bytes(
            pr.n, pr.m, pr.d, lds._flags(args.precision))))
        aws = lds.Workspace(lds.workspace_bytes(pr.n, pr.m, pr.d, 128, args.precision))
        V = torch.randn(pr.m, 128, device="cuda")
        PV = torch.empty(pr.n, 128, device="cuda")
        for _ in range(args.profile_passes):
            lds.plan_diagnostics(X, Y, f, g, eps, precision=args.precision, workspace=dws,
                                 as_dict=False)
            lds.transport_apply(X, Y, f, g, eps, V, precision=args.precision, out=PV,
                                workspace=aws)
        torch.cuda.synchronize()
        if lds.workspace_status(dws) != 0 or lds.workspace_status(aws) != 0:
            raise RuntimeError("device timeout reported")
        extra = f", then {args.profile_passes} x (diagnostics + P V k=128)"
    torch.cuda.synchronize()
    if lds.workspace_status(ws) != 0:
        raise RuntimeError("device timeout reported")
    print(f"profile driver: n=m={pr.n} d={pr.d} {args.precision}: "
          f"{2 * args.profile_passes + 1} LSE passes{extra}, f[0]={float(f[0]):.6f}")


def run_measure_tf32_peak(args):
    """Dense tf32 tensor-core throughput of this GPU, measured like the bf16 peaks the
    roofline lines use: torch.matmul of two 8192 x 8192 fp32 matrices with tf32 allowed
    (2 N^3 flops), best of 10 single launches (burst) and back to back for 4 s under the
    power cap (sustained), CUDA events, SM clocks sampled during each."""
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    torch.set_float32_matmul_precision("high")  # allow tf32 tensor cores for fp32 matmul
    N = 8192
    gen = torch.Generator(device=dev).manual_seed(8192)
    A = torch.randn(N, N, device=dev, generator=gen)
    B = torch.randn(N, N, device=dev, generator=gen)
    C = torch.empty(N, N, device=dev)
    flops = 2.0 * N ** 3
    for _ in range(5):
        torch.matmul(A, B, out=C)
    torch.cuda.synchronize()
    err = float((C[:64, :64].double() - A[:64].double() @ B[:, :64].double()).abs().max())
    clocks = ClockSampler(0).start()
    time.sleep(0.3)
    best = float("inf")
    for _ in range(10):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(A, B, out=C)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    clk_burst = clocks.stop()
    reps = max(1, int(4.0 / (best / 1e3)))
    clocks = ClockSampler(0).start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        torch.matmul(A, B, out=C)
    e1.record()
    torch.cuda.synchronize()
    clk_sus = clocks.stop()
    ms = e0.elapsed_time(e1)
    rec = {"command": "python bench.py --measure-tf32-peak --write-peak",
           "tf32_tflops": flops / (best / 1e3) / 1e12,
           "tf32_tflops_sustained": flops * reps / (ms / 1e3) / 1e12,
           "how": "torch.matmul fp32 8192^3 with torch.set_float32_matmul_precision('high') "
                  "(tf32 tensor cores), 2*N^3 flops: best of 10 (burst) and %d back to back "
                  "(sustained, %.1f s), CUDA events" % (reps, ms / 1e3),
           "max_abs_err_vs_fp64_64x64": err,
           "clocks_burst": clk_burst, "clocks_sustained": clk_sus,
           "gpu_name": torch.cuda.get_device_name(0), "sms": device_sms(),
           "torch": torch.__version__,
           "when": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime())}
    print(json.dumps(rec), flush=True)
    if args.write_peak:
        with open(TF32_PEAK_FILE, "w") as fh:
            json.dump(rec, fh, indent=1)
            fh.write("\n")


def main():
    args = parse_args()
    if args.measure_tf32_peak:
        run_measure_tf32_peak(args)
        return
    if args.profile_passes > 0:
        args.precision = args.precision or "bf16"
        run_profile_driver(args)
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.drift:
        run_drift(args)
    elif args.hvp:
        run_hvp(args)
    elif args.hvp_sweep:
        run_hvp_sweep(args)
    elif args.sk:
        run_sk(args)
    elif args.tol is not None:
        run_convergence(args)
    elif (args.workload != WORKLOAD_IDX or args.divergence or args.diagnostics
          or args.schedule != "alternating"):
        run_other_workload(args)
    else:
        if args.precision is None:
            args.precision = "bf16"
        run_gpu(args)


if __name__ == "__main__":
    main()
