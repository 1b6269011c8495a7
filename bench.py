"""Benchmark of the ragged-dot hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one ragged-dot forward over one batch of the workload (default: the Mixtral-like bf16
forward, 16384 rows x K=4096 x N=14336, G=8). Inputs are seeded synthetic data resident in HBM;
the timed region covers exactly K steps bracketed by a barrier and a device synchronisation,
timed with CUDA events on the launching stream. The JSON line reports useful TFLOP/s
(F_useful = 2 * sum(group_sizes) * K * N, the padded-work model's useful FLOPs in "How to Scale
Your Model on AMD", ch. 6 "Grouped GEMM kernels for MoE"), its fraction of the measured dense
bf16 peak, the roofline of the dominant kernel, an end-to-end number through the public API
with host buffers, the oracle timed on the host cores, and the other workloads of the suite.

Multi-GPU: one process per GPU (torchrun); the path shards by independent problems, so every
rank runs its own replica with no collective in the data path ("scaling": "weak").

``--impl reference`` times the fp64 CPU oracle instead (the reference arm of this suite) on the
host cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import rdot_inputs as ri  # noqa: E402

L2_BYTES = 129 * 2 ** 20


# ----------------------------------------------------------------------------------- helpers
def useful_flops(gs, k, n) -> float:
    return 2.0 * float(np.sum(np.maximum(gs, 0))) * k * n


def issued_rows(gs, tile_m: int, half_tiles: bool) -> int:
    """Rows the MMAs of a forward cover: the padded-work model of "How to Scale Your Model on AMD",
    chapter 6 ("Grouped GEMM kernels for MoE"): each group's rows rounded up to whole row tiles of
    tile_m rows, with 128-row tiles at group ends where the CTA-pair kernel has them."""
    gs = np.maximum(np.asarray(gs, np.int64), 0)
    if half_tiles and tile_m == 256:
        r = gs % 256
        return int(((gs // 256) * 256 + np.where(r == 0, 0, np.where(r <= 128, 128, 256))).sum())
    return int((-(-gs // tile_m) * tile_m).sum())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "fwd_tc_kernel": ["group_gemm_gb300/csrc/fwd_tc.cu", "group_gemm_gb300/csrc/ptx.cuh",
                      "group_gemm_gb300/csrc/sched.cuh", "group_gemm_gb300/csrc/epilogue.cuh",
                      "group_gemm_gb300/csrc/pdl.cuh"],
    "fwd_tc2_kernel": ["group_gemm_gb300/csrc/fwd_tc2.cu", "group_gemm_gb300/csrc/ptx.cuh",
                       "group_gemm_gb300/csrc/sched.cuh", "group_gemm_gb300/csrc/epilogue.cuh",
                       "group_gemm_gb300/csrc/pdl.cuh"],
}


def ncu_traffic(kernel: str, workload: str, sources):
    """Per-launch DRAM bytes from the committed ncu summary, or None when absent or when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{kernel}:{workload}")
    if not e or e.get("source_hash") != kernel_source_hash(sources):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0:   # wait for the first sample
            time.sleep(0.01)
        self.lines.clear()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in list(self.lines):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ workloads
def make_forward_inputs(name, device, seed=0):
    import torch
    cfg = ri.CONFIGS[name]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes(name, seed)
    dt = torch.bfloat16 if cfg["in_dtype"] == "bf16" else torch.float32
    lhs = ri.device_normal((m, k), 1000 + seed, cfg["lhs"][1], device, dt)
    rhs = ri.device_normal((g, k, n), 2000 + seed, cfg["rhs"][1], device, dt)
    return cfg, gs, lhs, rhs


def aggregate_over_ranks(t_local: float, units_local: float, world: int, device=None):
    """Whole-job numbers from one rank's timing: the max of the ranks' elapsed times and the sum
    of the units they processed (replicas: every rank processes units_local). Returns
    (t_max, total_units / t_max). Uses the process group's backend (NCCL on GPUs, gloo on CPU)."""
    if world <= 1:
        return t_local, units_local / t_local
    import torch
    import torch.distributed as dist
    tt = torch.tensor([t_local, units_local], dtype=torch.float64, device=device)
    t_max = tt[:1].clone()
    dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    units = tt[1:].clone()
    dist.all_reduce(units, op=dist.ReduceOp.SUM)
    t_max = float(t_max.item())
    return t_max, float(units.item()) / t_max


def time_region(fn, steps, stream, barrier, per_step_ms=None):
    """Seconds for `steps` calls of fn between a barrier + synchronize on both sides, by CUDA
    events on `stream`. With a list for per_step_ms, an event after every call also yields each
    step's duration (events are recorded between launches; the GPU work is unchanged)."""
    import torch
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if per_step_ms is not None else None
    start.record(stream)
    for i in range(steps):
        fn()
        if marks is not None:
            marks[i].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    if marks is not None:
        prev = start
        for m in marks:
            per_step_ms.append(prev.elapsed_time(m))
            prev = m
    return start.elapsed_time(end) / 1e3   # seconds


def cpu_oracle_sample(name, gs, lhs_host, rhs_host, budget_s, batch=16):
    """Times the fp64 oracle on successive batches of rows until ~budget_s seconds; returns
    (useful FLOP/s, cores, description)."""
    import oracle
    cfg = ri.CONFIGS[name]
    k, n = cfg["k"], cfg["n"]
    oracle.build()
    cores = oracle.set_threads(0)
    off = np.concatenate([[0], np.cumsum(gs)])
    valid = np.arange(int(off[-1]))
    rng = np.random.default_rng(7)
    order = rng.permutation(valid)
    done, t_total, i = 0, 0.0, 0
    while t_total < budget_s and i < order.size:
        rows = np.sort(order[i:i + batch])
        i += batch
        t0 = time.perf_counter()
        oracle.forward_rows(lhs_host, rhs_host, gs, rows)
        t_total += time.perf_counter() - t0
        done += rows.size
    flops = 2.0 * done * k * n
    return flops / t_total, cores, f"{done} random valid rows of {name} (x full N), fp64, {t_total:.1f} s"


# ---------------------------------------------------------------------------- our arm
def bench_ours(args, rank, world, barrier):
    import torch
    import group_gemm_gb300 as gg

    gg.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    name = args.workload
    cfg, gs, lhs, rhs = make_forward_inputs(name, dev)
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    flops = useful_flops(gs, k, n)
    plan = gg.Plan(m, k, n, g, "forward", cfg["in_dtype"], cfg["out_dtype"], device=dev.index)
    kernel = "fwd_tc2_kernel" if plan.info["tile_m"] == 256 else "fwd_tc_kernel"
    gs_d = torch.from_numpy(gs).to(dev)
    out_dt = torch.bfloat16 if cfg["out_dtype"] == "bf16" else torch.float32
    out = torch.empty((m, n), dtype=out_dt, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    step_ms = []
    t = time_region(step, args.steps, stream, barrier, step_ms)
    clk = clocks.stop()
    status = plan.status()
    if status:
        raise RuntimeError(f"device status bits {status:#x} after the timed region")
    t_max, rate = aggregate_over_ranks(t, flops * args.steps, world, dev)
    per_step = t_max / args.steps
    value = rate / 1e12
    launch_s = t / args.steps
    achieved = flops / launch_s / 1e12
    median_ms = float(np.median(step_ms))   # of the same timed region, step by step

    # end to end through the public API: every step copies its activations and group sizes in
    # from pinned host memory and its output back out. The copies are pipelined the way a
    # serving loop would run them: stream s_in brings step i+1's inputs while s_cmp computes step
    # i and s_out returns step i-1's output (two device buffers per tensor, guarded by events).
    lhs_h = torch.empty(lhs.shape, dtype=lhs.dtype, pin_memory=True)
    lhs_h.copy_(lhs)
    gs_h = torch.from_numpy(gs.copy()).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    lhs_b = [torch.empty_like(lhs) for _ in range(2)]
    gs_b = [torch.empty_like(gs_d) for _ in range(2)]
    out_b = [out, torch.empty_like(out)]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(nsteps):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        main = torch.cuda.current_stream(dev)
        start.record(main)
        for st in (s_in, s_cmp, s_out):
            st.wait_event(start)
        for e in ev_cmp + ev_out:
            e.record(main)
        for i in range(nsteps + 2):
            if i < nsteps:                                   # inputs of step i
                b = i % 2
                s_in.wait_event(ev_cmp[b])
                with torch.cuda.stream(s_in):
                    lhs_b[b].copy_(lhs_h, non_blocking=True)
                    gs_b[b].copy_(gs_h, non_blocking=True)
                ev_in[b].record(s_in)
            if 1 <= i <= nsteps:                             # compute of step i-1
                b = (i - 1) % 2
                s_cmp.wait_event(ev_in[b])
                s_cmp.wait_event(ev_out[b])
                gg.rdot_forward(plan.handle, lhs_b[b], rhs, gs_b[b], out_b[b], plan.workspace, s_cmp)
                ev_cmp[b].record(s_cmp)
            if i >= 2:                                       # output of step i-2
                b = (i - 2) % 2
                s_out.wait_event(ev_cmp[b])
                with torch.cuda.stream(s_out):
                    out_h.copy_(out_b[b], non_blocking=True)
                ev_out[b].record(s_out)
        for st in (s_in, s_cmp, s_out):
            main.wait_stream(st)
        end.record(main)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3

    e2e_run(max(2, args.warmup))
    e2e_steps = max(3, min(args.steps, 50))
    barrier()
    t_e2e = e2e_run(e2e_steps)
    barrier()
    t_e2e, e2e_rate = aggregate_over_ranks(t_e2e, flops * e2e_steps, world, dev)
    e2e = {"value": round(e2e_rate / 1e12, 3), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(lhs.numel() * lhs.element_size() + gs_d.numel() * 4),
           "d2h_bytes_per_step": int(out.numel() * out.element_size()),
           "steps": e2e_steps,
           "note": "weights resident; each step copies its activations and group sizes in and its output "
                   "out, pipelined over three streams (copy-in, compute, copy-out)"}
    # a timed region of back-to-back launches lasting a quarter second or more runs at the
    # power-capped clock, like the driver's sustained GEMM loop; a shorter one compares with the
    # burst figure
    if per_step * args.steps >= 0.25:
        peak, peak_kind = peaks["bf16_tflops_sustained"], f"{peaks['source']} bf16 sustained (timed region {per_step * args.steps:.2f} s)"
    else:
        peak, peak_kind = peaks["bf16_tflops"], f"{peaks['source']} bf16 burst (timed region {per_step * args.steps:.3f} s)"
    tile_m, tile_n = int(plan.info["tile_m"]), int(plan.info["tile_n"])
    w_pad = issued_rows(gs, tile_m, tile_m == 256 and tile_n != 512) / max(1.0, float(np.maximum(gs, 0).sum())) - 1.0
    result = {
        "metric": "ragged-dot useful TFLOP/s (fraction of GB300 dense bf16 peak; speedup vs padded in per_config)",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 4),
        "ms_per_step_median": round(median_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg["in_dtype"], "data": "synthetic (seeded)",
        "config": {"workload": f"{name}: M={m} K={k} N={n} G={g}, {cfg['in_dtype']} in / {cfg['out_dtype']} out",
                   "group_sizes": f"sum={int(gs.sum())} min={int(gs.min())} max={int(gs.max())}",
                   "l2": "inputs larger than L2 (no flush)" if (lhs.numel() * lhs.element_size() + rhs.numel()
                                                               * rhs.element_size()) > L2_BYTES else "warm L2",
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": round(value / world / peaks["bf16_tflops"], 4),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": ncu_traffic(kernel, name, KERNEL_SOURCES[kernel]),
                     "kernel": kernel, "tile": f"{plan.info['tile_m']}x{plan.info['tile_n']}",
                     "peak_kind": peak_kind,
                     "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
                     # tile tails: issued rows / useful rows - 1, and the issued MMA work against the peak
                     "w_pad": round(w_pad, 4), "issued_frac": round(achieved * (1.0 + w_pad) / peak, 4)},
        "e2e": e2e,
        "gpu_launches": args.steps,   # one librdot launch per timed step
        "clocks": clk,
        "device_status": status,
    }
    if rank == 0 and not args.no_extras:
        result["sustained"] = sustained_region(step, stream, dev, flops, per_step, peaks, kernel)
    del lhs, rhs, out, lhs_h, out_h, lhs_b, out_b, gs_b
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_extras and name != "deepseek_bf16":
        result["target_config"] = hbm_bound_forward("deepseek_bf16", dev, args.steps, peaks)
    if rank == 0 and not args.no_extras:
        try:
            result["per_config"] = extra_configs(args, dev, peaks, name, launch_s)
        except Exception as e:  # a failing extra must not hide the main line
            result["per_config"] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_leg(name, args.cpu_seconds)
    return result


def sustained_region(step, stream, dev, flops, burst_step_s, peaks, kernel, seconds=0.6):
    """The headline kernel over a back-to-back region of at least half a second, where the GPU
    settles at its power-capped clock (as in the sustained cuBLAS loop of the peak file): the mean
    launch time, the median SM clock sampled during the region, time x median clock (the clock
    cycles a launch takes, comparable between regions run at different clocks) and the fraction of
    the measured sustained bf16 peak."""
    steps = max(50, int(seconds / max(burst_step_s, 1e-6)))
    for _ in range(3):
        step()
    clocks = ClockSampler(dev.index)
    clocks.start()
    t = time_region(step, steps, stream, lambda: None)
    clk = clocks.stop()
    launch_s = t / steps
    achieved = flops / launch_s / 1e12
    mhz = clk.get("sm_mhz")
    return {"kernel": kernel, "steps": steps, "region_s": round(t, 3), "ms": round(launch_s * 1e3, 4),
            "tflops": round(achieved, 3), "peak": peaks["bf16_tflops_sustained"],
            "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
            "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
            "sm_mhz_median": mhz, "reasons": clk.get("reasons"),
            "mcycles_per_launch": round(launch_s * 1e3 * mhz / 1e3, 4) if mhz else None,
            "burst_ms": round(burst_step_s * 1e3, 4)}


def hbm_bound_forward(name, dev, steps, peaks):
    """The DeepSeek-like bf16 forward (256 fine-grained experts, Zipf-skewed routing), the
    configuration whose target is stated as a fraction of the dense bf16 peak. Every non-empty
    expert's weights must cross HBM once, so the launch is bound by HBM, not by the tensor cores:
    the roofline object reports the algorithmic bytes (lhs rows + weights of the non-empty groups
    + output) per second against the measured copy bandwidth, and beside it the useful TFLOP/s as a
    fraction of the bf16 peak together with the largest fraction that HBM bound allows."""
    import torch
    import group_gemm_gb300 as gg
    cfg, gs, lhs, rhs = make_forward_inputs(name, dev)
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    plan = gg.Plan(m, k, n, g, "forward", cfg["in_dtype"], cfg["out_dtype"], device=dev.index)
    kernel = "fwd_tc2_kernel" if plan.info["tile_m"] == 256 else "fwd_tc_kernel"
    gs_d = torch.from_numpy(gs).to(dev)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = max(10, min(steps, 100))

    def step():
        gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, stream)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    t = time_region(step, steps, stream, lambda: None)
    clk = clocks.stop()
    launch_s = t / steps
    fl = useful_flops(gs, k, n)
    nz = int(np.count_nonzero(gs))
    alg_bytes = (nz * k * n + int(gs.sum()) * k + m * n) * 2
    achieved = alg_bytes / launch_s / 1e9
    attainable = fl / (alg_bytes / (peaks["hbm_gbs"] * 1e9)) / 1e12
    res = {"workload": f"{name}: M={m} K={k} N={n} G={g} ({nz} non-empty), bf16 in / bf16 out",
           "ms": round(launch_s * 1e3, 4), "steps": steps, "tflops": round(fl / launch_s / 1e12, 3),
           "frac_of_bf16_peak": round(fl / launch_s / 1e12 / peaks["bf16_tflops"], 4),
           "attainable_frac_of_bf16_peak": round(attainable / peaks["bf16_tflops"], 4),
           "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": round(achieved / peaks["hbm_gbs"], 4),
                        "traffic": ncu_traffic(kernel, name, KERNEL_SOURCES[kernel]),
                        "algorithmic_bytes": alg_bytes, "kernel": kernel,
                        "tile": f"{plan.info['tile_m']}x{plan.info['tile_n']}"},
           "clocks": clk, "status": plan.status()}
    del lhs, rhs, out
    torch.cuda.empty_cache()
    return res


def _time_steps(fn, steps, stream):
    for _ in range(3):
        fn()
    return time_region(fn, steps, stream, lambda: None) / steps


def _time_graph(fn, dev, calls=20, replays=5):
    """Device time of one call of fn(stream): `calls` calls captured in a CUDA graph on a side
    stream, replayed `replays` times between CUDA events (no host launch cost in the region)."""
    import torch
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            fn(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(calls):
            fn(side)
    cur = torch.cuda.current_stream(dev)
    g.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    for _ in range(replays):
        g.replay()
    b.record(cur)
    torch.cuda.synchronize(dev)
    del g
    return a.elapsed_time(b) / 1e3 / (calls * replays)


def measure_fp8_peak(dev, n=8192, reps=10):
    """Dense FP8 tensor-core throughput on this GPU through torch._scaled_mm (E4M3 x E4M3 -> bf16,
    n^3, best of `reps` after warm-up): cuBLAS's MXFP8 GEMM (E8M0 scales, one per 32 elements of
    K: the block-scaled MMA the MXFP8 path issues) where torch offers it, else the GEMM with
    unit tensorwise scales. Returns (TFLOP/s, kind), or (None, None) where neither call works."""
    import torch
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()      # column-major operand
    except Exception:
        return None, None
    one = torch.ones((), device=dev, dtype=torch.float32)
    forms = []
    e8m0 = getattr(torch, "float8_e8m0fnu", None)
    if e8m0 is not None:
        sc = torch.full((n * (n // 32),), 127, dtype=torch.uint8, device=dev).view(e8m0)   # 2^0 everywhere
        forms.append(("cuBLAS MXFP8 GEMM (E8M0 block scales)", sc, sc))
    forms.append(("cuBLAS E4M3 GEMM (tensorwise scales)", one, one))
    result = (None, None)
    for kind, sa, sb in forms:
        try:
            def run():
                return torch._scaled_mm(a, b, scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)
            for _ in range(3):
                run()
            torch.cuda.synchronize(dev)
            best = float("inf")
            for _ in range(reps):
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record()
                run()
                e.record()
                e.synchronize()
                best = min(best, s.elapsed_time(e) / 1e3)
            result = (2.0 * n ** 3 / best / 1e12, f"measured here: {kind} {n}^3, best of {reps}")
            break
        except Exception:
            continue
    del a, b
    torch.cuda.empty_cache()
    return result


def extra_configs(args, dev, peaks, main_name, main_step_s):
    """The other workloads of the suite, measured the same way with fewer steps: the bf16
    forwards (with the padded-dense baseline beside them), the weight gradient and MXFP8."""
    import torch
    import group_gemm_gb300 as gg
    res = {}
    stream = torch.cuda.current_stream(dev)
    steps = max(5, min(args.steps, 30))
    for name in ("mixtral_bf16", "deepseek_bf16"):
        cfg, gs, lhs, rhs = make_forward_inputs(name, dev)
        m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
        plan = gg.Plan(m, k, n, g, "forward", cfg["in_dtype"], cfg["out_dtype"], device=dev.index)
        gs_d = torch.from_numpy(gs).to(dev)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        fl = useful_flops(gs, k, n)
        entry = {}
        if name == main_name:
            # the same kernel timed like the baselines below (a short burst), so that the
            # speedups compare like with like; the long timed region's figure is the bench value
            t = _time_steps(lambda: gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, stream),
                            steps, stream)
            entry["ms_burst"] = round(t * 1e3, 4)
        if name != main_name:
            t = _time_steps(lambda: gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, stream),
                            steps, stream)
            entry["tile"] = f"{plan.info['tile_m']}x{plan.info['tile_n']}"
            other = gg.Plan(m, k, n, g, "forward", cfg["in_dtype"], cfg["out_dtype"], device=dev.index,
                            flags=gg.RDOT_FLAG_NO_CTA_PAIR if plan.info["tile_m"] == 256 else gg.RDOT_FLAG_CTA_PAIR)
            t2 = _time_steps(lambda: gg.rdot_forward(other.handle, lhs, rhs, gs_d, out, other.workspace, stream),
                             steps, stream)
            entry["other_tile"] = {"tile": f"{other.info['tile_m']}x{other.info['tile_n']}",
                                   "tflops": round(fl / t2 / 1e12, 3), "ms": round(t2 * 1e3, 4)}
            nz = int(np.count_nonzero(gs))
            min_bytes = (nz * k * n + int(gs.sum()) * k + m * n) * 2
            entry.update({"tflops": round(fl / t / 1e12, 3), "ms": round(t * 1e3, 4),
                          "frac_of_bf16_peak": round(fl / t / 1e12 / peaks["bf16_tflops"], 4),
                          "hbm_gbs_algorithmic": round(min_bytes / t / 1e9, 1),
                          "frac_of_hbm": round(min_bytes / t / 1e9 / peaks["hbm_gbs"], 4)})
        # padded-dense baseline: every group padded to the largest group (rounded up to 128 rows)
        cap = -(-int(gs.max()) // 128) * 128
        pad = torch.empty(gg.rdot_padded_workspace_size(plan.handle, cap), dtype=torch.uint8, device=dev)
        tp = _time_steps(lambda: gg.rdot_padded_forward(plan.handle, lhs, rhs, gs_d, out, cap, pad, plan.workspace,
                                                        stream), max(3, steps // 5), stream)
        entry.update({"padded_ms": round(tp * 1e3, 3), "padded_tflops_useful": round(fl / tp / 1e12, 3),
                      "padded_capacity": cap, "padded_flops_ratio": round(g * cap / float(gs.sum()), 3)})
        entry["speedup_vs_padded"] = round(tp / t, 3)
        # the padded baseline's GEMM alone: the same kernel family on the padded buffers that the
        # call above left in its scratch (every group exactly `cap` rows), scatter/gather excluded
        rows = g * cap
        out_off = -(-rows * k * 2 // 256) * 256
        lhs_pad = pad[: rows * k * 2].view(torch.bfloat16).view(rows, k)
        out_pad = pad[out_off: out_off + rows * n * 2].view(torch.bfloat16).view(rows, n)
        uni = gg.Plan(rows, k, n, g, "forward", "bf16", "bf16", device=dev.index,
                      flags=gg.RDOT_FLAG_CTA_PAIR if plan.info["tile_m"] == 256 else gg.RDOT_FLAG_NO_CTA_PAIR)
        gs_u = torch.full((g,), cap, dtype=torch.int32, device=dev)
        tg = _time_steps(lambda: gg.rdot_forward(uni.handle, lhs_pad, rhs, gs_u, out_pad, uni.workspace, stream),
                         max(3, steps // 5), stream)
        entry.update({"padded_gemm_only_ms": round(tg * 1e3, 3), "speedup_vs_padded_gemm_only": round(tg / t, 3)})
        entry["status"] = plan.status()
        res[name] = entry
        del lhs, rhs, out, pad
        torch.cuda.empty_cache()
    # decode-sized forwards: a few dozen tokens, or a single one, so every routed expert's weights
    # stream once (HBM-bound whatever the tile shape: a tile's MMAs on its few valid rows take less
    # time than its weight slab takes to arrive); reported against the HBM copy peak
    for name, tokens, topk, sigma, key in (("mixtral_bf16", 64, 2, None, "decode_mixtral_bf16"),
                                           ("deepseek_bf16", 64, 8, 1.1, "decode_deepseek_bf16"),
                                           ("mixtral_bf16", 1, 2, None, "decode_mixtral_bf16_t1"),
                                           ("deepseek_bf16", 1, 8, 1.1, "decode_deepseek_bf16_t1"),
                                           ("deepseek_bf16", 8, 8, 1.1, "decode_deepseek_bf16_t8")):
        cfg = ri.CONFIGS[name]
        k, n, g = cfg["k"], cfg["n"], cfg["g"]
        gs = (ri.routed_group_sizes(tokens, g, topk, 1.0, seed=0) if sigma is None else
              ri.zipf_routed_group_sizes(tokens, g, topk, sigma, seed=0, n_zero=8))
        m = int(gs.sum())
        lhs = ri.device_normal((m, k), 1, 1.0, dev, torch.bfloat16)
        rhs = ri.device_normal((g, k, n), 2, 0.02, dev, torch.bfloat16)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        gs_d = torch.from_numpy(gs).to(dev)
        plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16", device=dev.index)
        t = _time_steps(lambda: gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, stream), 20, stream)
        wbytes = int(np.count_nonzero(gs)) * k * n * 2 + m * (k + n) * 2
        res[key] = {"workload": f"{tokens} tokens top-{topk}: M={m}, {int(np.count_nonzero(gs))} of {g} "
                                f"experts routed", "ms": round(t * 1e3, 4),
                    "hbm_gbs_algorithmic": round(wbytes / t / 1e9, 1),
                    "frac_of_hbm": round(wbytes / t / 1e9 / peaks["hbm_gbs"], 4), "status": plan.status(),
                    "tile": f"{plan.info['tile_m']}x{plan.info['tile_n']}"}
        if plan.info["tile_m"] < 128:
            # the plan took the swapped small-row kernel; the row-tile kernels on the same call
            rp = gg.Plan(m, k, n, g, "forward", "bf16", "bf16", flags=gg.RDOT_FLAG_NO_SKINNY, device=dev.index)
            tr = _time_steps(lambda: gg.rdot_forward(rp.handle, lhs, rhs, gs_d, out, rp.workspace, stream), 20,
                             stream)
            res[key]["ms_row_tiles"] = round(tr * 1e3, 4)
            res[key]["tile_row_tiles"] = f"{rp.info['tile_m']}x{rp.info['tile_n']}"
        del lhs, rhs, out
        torch.cuda.empty_cache()
    # data gradient of the Mixtral-like forward: dlhs [M, K] = dy [M, N] . rhs[g]^T
    cfg = ri.CONFIGS["mixtral_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("mixtral_bf16")
    dy = ri.device_normal((m, n), 3000, 1.0, dev, torch.bfloat16)
    rhs = ri.device_normal((g, k, n), 2000, 0.02, dev, torch.bfloat16)
    dlhs = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
    gs_d = torch.from_numpy(gs).to(dev)
    plan = gg.Plan(m, k, n, g, "grad_input", "bf16", "bf16", device=dev.index)
    t = _time_steps(lambda: gg.rdot_grad_input(plan.handle, dy, rhs, gs_d, dlhs, plan.workspace, stream), steps,
                    stream)
    fl = useful_flops(gs, k, n)
    res["dgrad_bf16"] = {"workload": f"data gradient of mixtral_bf16: dy [{m}, {n}] x rhs [{g}, {k}, {n}] -> [{m}, {k}]",
                         "tflops": round(fl / t / 1e12, 3), "ms": round(t * 1e3, 4),
                         "frac_of_bf16_peak": round(fl / t / 1e12 / peaks["bf16_tflops"], 4), "status": plan.status(),
                         "tile": f"{plan.info['tile_m']}x{plan.info['tile_n']}"}
    del dy, rhs, dlhs
    torch.cuda.empty_cache()
    # fused gated up projection at the Mixtral-like size: silu(x w0) * (x w1), two ragged dots
    x = ri.device_normal((m, k), 1000, 1.0, dev, torch.bfloat16)
    rhs1 = ri.device_normal((g, k, n), 2001, 0.02, dev, torch.bfloat16)
    rhs0 = ri.device_normal((g, k, n), 2000, 0.02, dev, torch.bfloat16)
    hout = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    plan = gg.Plan(m, k, n, g, "forward_gated", "bf16", "bf16", device=dev.index)
    t = _time_steps(lambda: gg.rdot_forward_gated(plan.handle, x, rhs0, rhs1, gs_d, hout, plan.workspace, stream),
                    steps, stream)
    fl = 2.0 * useful_flops(gs, k, n)
    res["gated_up_bf16"] = {"workload": f"silu(x w0) * (x w1): x [{m}, {k}], w0/w1 [{g}, {k}, {n}]",
                            "tflops": round(fl / t / 1e12, 3), "ms": round(t * 1e3, 4),
                            "frac_of_bf16_peak": round(fl / t / 1e12 / peaks["bf16_tflops"], 4),
                            "status": plan.status(), "tile": "256x128 (x2 accumulators: w0, w1)"}
    del x, rhs0, rhs1, hout
    torch.cuda.empty_cache()
    # a whole Mixtral-like expert layer on the library: permute -> gated up projection -> down
    # projection -> weighted un-permute (8192 tokens, top-2 of 8, 4096 -> 14336 -> 4096)
    t_l, k_l = m // 2, 2
    rng = np.random.default_rng(1)
    ids_l = torch.from_numpy(np.argsort(-rng.standard_normal((t_l, g)), axis=1)[:, :k_l].astype(np.int32)).to(dev)
    wr_l = torch.rand((t_l, k_l), device=dev)
    x_l = ri.device_normal((t_l, k), 5000, 1.0, dev, torch.bfloat16)
    w0_l = ri.device_normal((g, k, n), 5001, 0.02, dev, torch.bfloat16)
    w1_l = ri.device_normal((g, k, n), 5002, 0.02, dev, torch.bfloat16)
    wo_l = ri.device_normal((g, n, k), 5003, 0.02, dev, torch.bfloat16)

    def layer():
        xs_l, gs_l, _, inv_l = gg.moe_permute(ids_l, x_l, g, stream)
        h_l = gg.ragged_dot_gated(xs_l, w0_l, w1_l, gs_l, stream=stream)
        y_l = gg.ragged_dot(h_l, wo_l, gs_l, stream=stream)
        return gg.moe_unpermute(y_l, inv_l, wr_l, stream=stream)
    tl = _time_steps(layer, max(5, steps // 3), stream)
    fl_l = 3.0 * 2.0 * t_l * k_l * k * n
    res["moe_layer"] = {"workload": f"{t_l} tokens top-{k_l} of {g}: permute, gated up {k}->{n}, down {n}->{k}, "
                                    "un-permute", "ms": round(tl * 1e3, 4), "tflops": round(fl_l / tl / 1e12, 3),
                        "frac_of_bf16_peak": round(fl_l / tl / 1e12 / peaks["bf16_tflops"], 4),
                        "launches_per_layer": 4 + 1 + 1 + 1}

    # the same layer with the weighted un-permute fused into the down projection's epilogue
    # (fp32 [T, N] out, cleared by a memset, each copy's row added with fp32 reductions)
    def layer_fused():
        xs_l, gs_l, order_l, _ = gg.moe_permute(ids_l, x_l, g, stream)
        h_l = gg.ragged_dot_gated(xs_l, w0_l, w1_l, gs_l, stream=stream)
        return gg.ragged_dot_combine(h_l, wo_l, gs_l, order_l, wr_l, stream=stream)
    # the two layers alternate in rounds, so that both see the same power-capped clock drift
    t_un, t_fu = [], []
    for _ in range(5):
        t_un.append(_time_steps(layer, max(3, steps // 6), stream))
        t_fu.append(_time_steps(layer_fused, max(3, steps // 6), stream))
    tl, tlf = float(np.median(t_un)), float(np.median(t_fu))
    res["moe_layer"].update({"ms": round(tl * 1e3, 4), "tflops": round(fl_l / tl / 1e12, 3),
                             "frac_of_bf16_peak": round(fl_l / tl / 1e12 / peaks["bf16_tflops"], 4),
                             "timing": "median of 5 rounds alternating with the fused layer"})
    # the down projection step alone, both ways: ragged dot + un-permute vs the fused call
    xs_l, gs_l, order_l, inv_l = gg.moe_permute(ids_l, x_l, g, stream)
    h_l = gg.ragged_dot_gated(xs_l, w0_l, w1_l, gs_l, stream=stream)
    y_l = torch.empty((t_l * k_l, k), dtype=torch.bfloat16, device=dev)
    o_l = torch.empty((t_l, k), dtype=torch.bfloat16, device=dev)
    of_l = torch.empty((t_l, k), dtype=torch.float32, device=dev)
    t_dn, t_df = [], []
    for _ in range(5):
        t_dn.append(_time_steps(lambda: (gg.ragged_dot(h_l, wo_l, gs_l, out=y_l, stream=stream),
                                         gg.moe_unpermute(y_l, inv_l, wr_l, out=o_l, stream=stream)),
                                max(3, steps // 3), stream))
        t_df.append(_time_steps(lambda: gg.ragged_dot_combine(h_l, wo_l, gs_l, order_l, wr_l, out=of_l,
                                                              stream=stream), max(3, steps // 3), stream))
    t_down, t_down_fused = float(np.median(t_dn)), float(np.median(t_df))
    res["moe_layer_fused_combine"] = {
        "workload": res["moe_layer"]["workload"] + "; un-permute fused into the down projection (fp32 out)",
        "ms": round(tlf * 1e3, 4), "tflops": round(fl_l / tlf / 1e12, 3),
        "frac_of_bf16_peak": round(fl_l / tlf / 1e12 / peaks["bf16_tflops"], 4),
        "launches_per_layer": 4 + 1 + 1 + 1, "speedup_vs_unfused_layer": round(tl / tlf, 4),
        "down_plus_unpermute_ms": round(t_down * 1e3, 4), "down_fused_combine_ms": round(t_down_fused * 1e3, 4)}
    del xs_l, h_l, y_l, o_l, of_l
    del x_l, w0_l, w1_l, wo_l
    torch.cuda.empty_cache()
    # MoE permute / un-permute around the Mixtral-like layer: 8192 tokens, top-2 of 8, width 4096
    t, k, e, width = m // 2, 2, g, cfg["k"]
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((t, e))
    ids = torch.from_numpy(np.argsort(-logits, axis=1)[:, :k].astype(np.int32)).to(dev)
    x = ri.device_normal((t, width), 4000, 1.0, dev, torch.bfloat16)
    xs = torch.empty((t * k, width), dtype=torch.bfloat16, device=dev)
    gsz = torch.empty(e, dtype=torch.int32, device=dev)
    order = torch.empty(t * k, dtype=torch.int32, device=dev)
    inv = torch.empty(t * k, dtype=torch.int32, device=dev)
    ws = torch.empty(gg.rdot_moe_route_workspace_size(t, k, e), dtype=torch.uint8, device=dev)
    tp_loop = _time_steps(lambda: gg.rdot_moe_permute(ids, x, e, gsz, order, inv, xs, ws, stream), steps, stream)
    tp = _time_graph(lambda st: gg.rdot_moe_permute(ids, x, e, gsz, order, inv, xs, ws, st), dev)
    wr = torch.rand((t, k), device=dev)
    outc = torch.empty((t, width), dtype=torch.bfloat16, device=dev)
    tc_loop = _time_steps(lambda: gg.rdot_moe_unpermute(xs, inv, wr, outc, stream), steps, stream)
    tc = _time_graph(lambda st: gg.rdot_moe_unpermute(xs, inv, wr, outc, st), dev)
    perm_bytes = t * width * 2 + t * k * width * 2 + t * k * 4 * 3 + e * 4      # x once, x_sorted, ids/order/inv
    comb_bytes = t * k * width * 2 + t * width * 2 + t * k * 8                  # y_sorted, out, inv + weights
    res["moe_route"] = {"workload": f"{t} tokens, top-{k} of {e} experts, rows of {width} bf16",
                        "timing": "device time per call from CUDA-graph replays of 20 calls; *_python_loop: "
                                  "one Python call per step, host launch cost included",
                        "permute_ms": round(tp * 1e3, 4), "permute_gbs_algorithmic": round(perm_bytes / tp / 1e9, 1),
                        "permute_frac_of_hbm": round(perm_bytes / tp / 1e9 / peaks["hbm_gbs"], 4),
                        "permute_ms_python_loop": round(tp_loop * 1e3, 4),
                        "unpermute_ms": round(tc * 1e3, 4), "unpermute_gbs_algorithmic": round(comb_bytes / tc / 1e9, 1),
                        "unpermute_frac_of_hbm": round(comb_bytes / tc / 1e9 / peaks["hbm_gbs"], 4),
                        "unpermute_ms_python_loop": round(tc_loop * 1e3, 4)}
    del x, xs, outc, ws
    torch.cuda.empty_cache()
    # router top-k (the front end): Mixtral-like 8192 tokens x 8 experts top-2, DeepSeek-like 4096
    # tokens x 256 experts top-8, fp32 logits N(0, 1), softmax weights; a few MB per call, so the
    # launch's latency rather than HBM bandwidth bounds it
    res["router_topk"] = {}
    for tt, ee, kk in ((8192, 8, 2), (4096, 256, 8)):
        lg = ri.device_normal((tt, ee), 4100 + ee, 1.0, dev, torch.float32)
        ids_t = torch.empty((tt, kk), dtype=torch.int32, device=dev)
        w_t = torch.empty((tt, kk), dtype=torch.float32, device=dev)
        tr = _time_graph(lambda st: gg.rdot_router_topk(lg, kk, gg.RDOT_ROUTER_SOFTMAX, ids_t, w_t, st), dev)
        rb = tt * ee * 4 + tt * kk * 8
        res["router_topk"][f"T{tt}_E{ee}_k{kk}"] = {"us": round(tr * 1e6, 2), "bytes": rb,
                                                    "hbm_gbs_algorithmic": round(rb / tr / 1e9, 1),
                                                    "frac_of_hbm": round(rb / tr / 1e9 / peaks["hbm_gbs"], 4)}
        del lg, ids_t, w_t
    # weight gradient
    cfg = ri.CONFIGS["wgrad_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("wgrad_bf16")
    lhs = ri.device_normal((m, k), 1000, 1.0, dev, torch.bfloat16)
    dy = ri.device_normal((m, n), 2000, 1.0, dev, torch.bfloat16)
    dw = torch.empty((g, k, n), dtype=torch.float32, device=dev)
    plan = gg.Plan(m, k, n, g, "grad_weight", "bf16", "f32", device=dev.index)
    gs_d = torch.from_numpy(gs).to(dev)
    t = _time_steps(lambda: gg.rdot_grad_weight(plan.handle, lhs, dy, gs_d, dw, plan.workspace, stream), steps,
                    stream)
    fl = useful_flops(gs, k, n)
    min_bytes = 2 * m * (k + n) + 4 * g * k * n
    res["wgrad_bf16"] = {"tflops": round(fl / t / 1e12, 3), "ms": round(t * 1e3, 4),
                         "frac_of_bf16_peak": round(fl / t / 1e12 / peaks["bf16_tflops"], 4),
                         "hbm_gbs_algorithmic": round(min_bytes / t / 1e9, 1), "status": plan.status(),
                         "tile": f"{plan.info['tile_m']}x{plan.info['tile_n']}"}
    other = gg.Plan(m, k, n, g, "grad_weight", "bf16", "f32", device=dev.index,
                    flags=gg.RDOT_FLAG_NO_CTA_PAIR if plan.info["tile_m"] == 256 else gg.RDOT_FLAG_CTA_PAIR)
    t2 = _time_steps(lambda: gg.rdot_grad_weight(other.handle, lhs, dy, gs_d, dw, other.workspace, stream), steps,
                     stream)
    res["wgrad_bf16"]["other_tile"] = {"tile": f"{other.info['tile_m']}x{other.info['tile_n']}",
                                       "tflops": round(fl / t2 / 1e12, 3), "ms": round(t2 * 1e3, 4)}
    # the same weight gradient with a bf16 dw (the output type of the pages' wgrad_wi example)
    dwh = torch.empty((g, k, n), dtype=torch.bfloat16, device=dev)
    ph = gg.Plan(m, k, n, g, "grad_weight", "bf16", "bf16", device=dev.index)
    t3 = _time_steps(lambda: gg.rdot_grad_weight(ph.handle, lhs, dy, gs_d, dwh, ph.workspace, stream), steps, stream)
    min_bytes_h = 2 * m * (k + n) + 2 * g * k * n
    res["wgrad_bf16"]["dw_bf16"] = {"tflops": round(fl / t3 / 1e12, 3), "ms": round(t3 * 1e3, 4),
                                    "frac_of_bf16_peak": round(fl / t3 / 1e12 / peaks["bf16_tflops"], 4),
                                    "hbm_gbs_algorithmic": round(min_bytes_h / t3 / 1e9, 1), "status": ph.status(),
                                    "tile": f"{ph.info['tile_m']}x{ph.info['tile_n']}"}
    del lhs, dy, dw, dwh
    torch.cuda.empty_cache()
    # MXFP8 forward
    cfg = ri.CONFIGS["mxfp8"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("mxfp8")
    x = ri.device_normal((m, k), 1000, 1.0, dev, torch.float32)
    aq, as_ = ri.quantize_mx_e4m3(x, axis=1)
    del x
    w = ri.device_normal((g, k, n), 2000, 0.02, dev, torch.float32)
    bq, bs = ri.quantize_mx_e4m3(w, axis=1)
    del w
    torch.cuda.empty_cache()
    plan = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16", device=dev.index)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    gs_d = torch.from_numpy(gs).to(dev)
    t = _time_steps(lambda: gg.rdot_forward_mxfp8(plan.handle, aq, as_, bq, bs, gs_d, out, plan.workspace, stream),
                    steps, stream)
    fl = useful_flops(gs, k, n)
    fp8_measured, fp8_kind = measure_fp8_peak(dev)
    fp8_peak = fp8_measured if fp8_measured else 2.0 * peaks["bf16_tflops"]
    min_bytes = m * k + g * k * n + (m * k + g * k * n) // 32 + 2 * m * n
    res["mxfp8"] = {"tflops": round(fl / t / 1e12, 3), "ms": round(t * 1e3, 4),
                    "frac_of_fp8_peak": round(fl / t / 1e12 / fp8_peak, 4),
                    "fp8_peak_tflops": round(fp8_peak, 1),
                    "fp8_peak_kind": (fp8_kind if fp8_measured
                                      else "not measurable here; taken as 2x the measured bf16 burst peak"),
                    "hbm_gbs_algorithmic": round(min_bytes / t / 1e9, 1), "status": plan.status(),
                    "tile": f"{plan.info['tile_m']}x{plan.info['tile_n']}"}
    other = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16", device=dev.index,
                    tile_n=128 if plan.info["tile_n"] == 256 else 256)
    t2 = _time_steps(lambda: gg.rdot_forward_mxfp8(other.handle, aq, as_, bq, bs, gs_d, out, other.workspace, stream),
                     steps, stream)
    res["mxfp8"]["other_tile"] = {"tile": f"{other.info['tile_m']}x{other.info['tile_n']}",
                                  "tflops": round(fl / t2 / 1e12, 3), "ms": round(t2 * 1e3, 4)}
    pair = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16", device=dev.index,
                   flags=gg.RDOT_FLAG_NO_CTA_PAIR if plan.info["tile_m"] == 256 else gg.RDOT_FLAG_CTA_PAIR)
    t3 = _time_steps(lambda: gg.rdot_forward_mxfp8(pair.handle, aq, as_, bq, bs, gs_d, out, pair.workspace, stream),
                     steps, stream)
    # the data gradient on MXFP8 operands at the same size: dy [M, N] x w [G, K, N] -> [M, K]
    dyf = ri.device_normal((m, n), 3000, 1.0, dev, torch.float32)
    dq, dsc = ri.quantize_mx_e4m3(dyf, axis=1)
    del dyf
    wf = ri.device_normal((g, k, n), 2000, 0.02, dev, torch.float32)
    wq, wsc = ri.quantize_mx_e4m3(wf, axis=2)
    del wf
    torch.cuda.empty_cache()
    dplan = gg.Plan(m, k, n, g, "grad_input_mxfp8", "e4m3", "bf16", device=dev.index)
    dws = torch.zeros(gg.rdot_workspace_size(dplan.handle), dtype=torch.uint8, device=dev)
    dout = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
    t4 = _time_steps(lambda: gg.rdot_grad_input_mxfp8(dplan.handle, dq, dsc, wq, wsc, gs_d, dout, dws, stream),
                     steps, stream)
    res["mxfp8_dgrad"] = {"workload": f"dy [{m}, {n}] x w [{g}, {k}, {n}] -> [{m}, {k}], scales along {n}",
                          "tflops": round(fl / t4 / 1e12, 3), "ms": round(t4 * 1e3, 4),
                          "frac_of_fp8_peak": round(fl / t4 / 1e12 / fp8_peak, 4),
                          "status": gg.rdot_read_status(dplan.handle, dws),
                          "tile": f"{dplan.info['tile_m']}x{dplan.info['tile_n']}"}
    del dq, dsc, wq, wsc, dout, dws
    res["mxfp8"]["other_pairing"] = {"tile": f"{pair.info['tile_m']}x{pair.info['tile_n']}",
                                     "tflops": round(fl / t3 / 1e12, 3), "ms": round(t3 * 1e3, 4),
                                     "status": pair.status()}
    del aq, as_, bq, bs, out
    torch.cuda.empty_cache()
    # MXFP8 weight gradient at the grad-weight workload's shape: E4M3 lhs and dy with E8M0 scales
    # along the rows, in blocks of 32 from each group's start; fp32 dw
    cfg = ri.CONFIGS["wgrad_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("wgrad_bf16")
    x = ri.device_normal((m, k), 1000, 1.0, dev, torch.float32)
    aq, as_ = ri.quantize_mx_e4m3_group_rows(x, gs)
    del x
    dy = ri.device_normal((m, n), 2000, 1.0, dev, torch.float32)
    dq, dsc = ri.quantize_mx_e4m3_group_rows(dy, gs)
    del dy
    dw = torch.empty((g, k, n), dtype=torch.float32, device=dev)
    wplan = gg.Plan(m, k, n, g, "grad_weight_mxfp8", "e4m3", "f32", device=dev.index)
    gs_d = torch.from_numpy(gs).to(dev)
    t5 = _time_steps(lambda: gg.rdot_grad_weight_mxfp8(wplan.handle, aq, as_, dq, dsc, gs_d, dw, wplan.workspace,
                                                       stream), steps, stream)
    fl = useful_flops(gs, k, n)
    min_bytes = m * (k + n) + (m // 32 + g) * (k + n) + 4 * g * k * n       # codes, scales, fp32 dw
    res["mxfp8_wgrad"] = {"workload": f"dw [{g}, {k}, {n}] from E4M3 lhs [{m}, {k}] and dy [{m}, {n}], scales "
                                      "along the rows per group", "tflops": round(fl / t5 / 1e12, 3),
                          "ms": round(t5 * 1e3, 4), "frac_of_fp8_peak": round(fl / t5 / 1e12 / fp8_peak, 4),
                          "hbm_gbs_algorithmic": round(min_bytes / t5 / 1e9, 1),
                          "frac_of_hbm": round(min_bytes / t5 / 1e9 / peaks["hbm_gbs"], 4),
                          "status": wplan.status(), "tile": f"{wplan.info['tile_m']}x{wplan.info['tile_n']}"}
    dwh = torch.empty((g, k, n), dtype=torch.bfloat16, device=dev)
    hplan = gg.Plan(m, k, n, g, "grad_weight_mxfp8", "e4m3", "bf16", device=dev.index)
    t6 = _time_steps(lambda: gg.rdot_grad_weight_mxfp8(hplan.handle, aq, as_, dq, dsc, gs_d, dwh, hplan.workspace,
                                                       stream), steps, stream)
    res["mxfp8_wgrad"]["dw_bf16"] = {"tflops": round(fl / t6 / 1e12, 3), "ms": round(t6 * 1e3, 4),
                                     "frac_of_fp8_peak": round(fl / t6 / 1e12 / fp8_peak, 4), "status": hplan.status()}
    del aq, as_, dq, dsc, dw, dwh
    torch.cuda.empty_cache()
    # MXFP8 forward at the MoE GEMM shape the AITER follow-ups time (E 32, N 2048, K 6144) with
    # T rows routed top-1 (the pages give neither the top-k nor the rows per call); the weights
    # of the routed experts stream once, so the figure is the fraction of the HBM copy peak
    e_, n_, k_ = 32, 2048, 6144
    wf = ri.device_normal((e_, k_, n_), 2, 0.02, dev, torch.float32)
    wq, wsc = ri.quantize_mx_e4m3(wf, axis=1)
    del wf
    dec = {}
    for tokens in (8, 64, 512, 2048):
        gs = ri.routed_group_sizes(tokens, e_, 1, 1.0, seed=0)
        m = int(gs.sum())
        xf = ri.device_normal((m, k_), 1, 1.0, dev, torch.float32)
        xq, xs = ri.quantize_mx_e4m3(xf, axis=1)
        del xf
        out = torch.empty((m, n_), dtype=torch.bfloat16, device=dev)
        gs_d = torch.from_numpy(gs).to(dev)
        nz = int(np.count_nonzero(gs))
        wbytes = nz * k_ * n_ + nz * (k_ // 32) * n_ + m * (k_ + k_ // 32) + 2 * m * n_
        plan = gg.Plan(m, k_, n_, e_, "forward_mxfp8", "e4m3", "bf16", device=dev.index)
        t = _time_steps(lambda: gg.rdot_forward_mxfp8(plan.handle, xq, xs, wq, wsc, gs_d, out, plan.workspace,
                                                      stream), 20, stream)
        entry = {"rows": m, "experts_routed": nz, "ms": round(t * 1e3, 4),
                 "frac_of_hbm": round(wbytes / t / 1e9 / peaks["hbm_gbs"], 4), "status": plan.status(),
                 "tile": f"{plan.info['tile_m']}x{plan.info['tile_n']}"}
        if plan.info["tile_m"] < 128:
            rp = gg.Plan(m, k_, n_, e_, "forward_mxfp8", "e4m3", "bf16", flags=gg.RDOT_FLAG_NO_SKINNY,
                         device=dev.index)
            tr = _time_steps(lambda: gg.rdot_forward_mxfp8(rp.handle, xq, xs, wq, wsc, gs_d, out, rp.workspace,
                                                           stream), 20, stream)
            entry["ms_row_tiles"] = round(tr * 1e3, 4)
        dec[f"T{tokens}"] = entry
        del xq, xs, out
    res["mxfp8_decode_e32_n2048_k6144"] = dec
    del wq, wsc
    torch.cuda.empty_cache()
    return res


def cpu_baseline_leg(name, seconds):
    import torch
    cfg = ri.CONFIGS[name]
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    if dev is not None:
        _, gs, lhs, rhs = make_forward_inputs(name, dev)
        lhs_h, rhs_h = lhs.cpu(), rhs.cpu()
        del lhs, rhs
        torch.cuda.empty_cache()
    else:
        gs = ri.config_group_sizes(name)
        lhs_h = torch.from_numpy(ri.host_normal((cfg["m"], cfg["k"]), 1000, cfg["lhs"][1])).to(torch.bfloat16)
        rhs_h = torch.from_numpy(ri.host_normal((cfg["g"], cfg["k"], cfg["n"]), 2000, cfg["rhs"][1])).to(torch.bfloat16)
    v, cores, sample = cpu_oracle_sample(name, gs, lhs_h, rhs_h, seconds)
    return {"value": round(v / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}


# ------------------------------------------------------------------------- reference arm
def bench_reference(args, rank, world):
    if rank != 0:
        return None
    import torch
    name = args.workload
    cfg = ri.CONFIGS[name]
    k, n = cfg["k"], cfg["n"]
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    if dev is not None:
        _, gs, lhs, rhs = make_forward_inputs(name, dev)
        lhs_h, rhs_h = lhs.cpu(), rhs.cpu()
        del lhs, rhs
        torch.cuda.empty_cache()
    else:
        gs = ri.config_group_sizes(name)
        std_l = cfg["lhs"][1] if cfg["lhs"][0] == "normal" else 1.0
        std_r = cfg["rhs"][1] if cfg["rhs"][0] == "normal" else 1.0
        lhs_h = torch.from_numpy(ri.host_normal((cfg["m"], cfg["k"]), 1000, std_l)).to(torch.bfloat16)
        rhs_h = torch.from_numpy(ri.host_normal((cfg["g"], k, n), 2000, std_r)).to(torch.bfloat16)
    import oracle
    oracle.build()
    cores = oracle.set_threads(0)
    # seconds of oracle work per step: the whole run stays near 150 s (a test may ask for less)
    per_step = getattr(args, "ref_step_seconds", None) or max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    rows_per_step = None
    for _ in range(args.warmup):
        v, _, _ = cpu_oracle_sample(name, gs, lhs_h, rhs_h, per_step)
        rows_per_step = rows_per_step or max(16, int(v * per_step / (2.0 * k * n)))
    rows_per_step = rows_per_step or 64
    off = int(np.sum(gs))
    rng = np.random.default_rng(11)
    t_total, fl_total = 0.0, 0.0
    for _ in range(args.steps):
        rows = np.sort(rng.choice(off, size=min(rows_per_step, off), replace=False))
        t0 = time.perf_counter()
        oracle.forward_rows(lhs_h, rhs_h, gs, rows)
        t_total += time.perf_counter() - t0
        fl_total += 2.0 * rows.size * k * n
    value = fl_total / t_total / 1e12
    sample = f"{rows_per_step} random valid rows of {name} (x full N) per step, fp64 oracle"
    return {
        "impl": "reference", "metric": "ragged-dot useful TFLOP/s (fraction of GB300 dense bf16 peak; speedup vs "
                                       "padded in per_config)",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_total / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": f"{name}: M={cfg['m']} K={k} N={n} G={cfg['g']}", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixtral_bf16", choices=["mixtral_bf16", "deepseek_bf16"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    barrier = lambda: None  # noqa: E731
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group(backend=backend)
        barrier = dist.barrier

    if args.impl == "reference":
        res = bench_reference(args, rank, world)
    else:
        res = bench_ours(args, rank, world, barrier)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
