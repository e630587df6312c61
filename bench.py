#!/usr/bin/env python3
"""Benchmark of the GB300 tiled GEMM library (D = A·Bᵀ, fp32 accumulate).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-extra]

One step is one GEMM of the chosen workload through the library's C ABI
(default: bf16 4096³, the compute-bound headline).  Inputs are seeded
synthetic data resident in HBM; before every timed step L2 is flushed (a
512 MiB write, then a 320 MiB read so the written lines are written back
outside the timing) unless the inputs alone exceed twice the L2, and the step
itself is timed with CUDA events on the launching stream.  Rank 0 prints ONE
JSON line.  Unless --no-extra is given, the line also carries a measurement
of every other workload: the "next" rows ("workloads", each with its own
roofline entry) and, as its last key, a compact block for the five
configurations C1-C5 ("configs": median time, throughput, roofline fraction,
kernel, and the CPU oracle timed on a bounded row sample of the same
configuration on the host cores).

--impl reference times the CPU oracle (oracle/, fp64, OpenMP on the host
cores) on bounded row samples of the same workload: the reference arm.
Under torchrun (N > 1) every rank runs its own replica of the workload on
its own GPU (weak scaling, no data-path collective); a gloo group is used
only for the barrier and the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s and % of GB300 dense tensor (or HBM) roofline, 1 GPU"
HEADLINE = "bf16_4096"
# the five configurations the metric is quoted on, in order (C1..C5)
CONFIGS = ("fp32_128", "bf16_1024", "bf16_4096", "skinny_16x28672x8192", "mxfp4_8192")
# seconds of oracle work per configuration in the compact per-configuration block
CONFIG_CPU_BUDGET = 3.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense ratios fp4 : bf16 and fp8 : bf16 on GB300 (13.5, 4.5 : 2.25 PFLOP/s)
FP4_OVER_BF16 = 13.5 / 2.25
FP8_OVER_BF16 = 4.5 / 2.25
# fp32 FFMA peak: 152 SMs x 128 FMA/clk x 2 flop x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
# GB300 nominal dense peaks (context beside the measured denominators)
NOMINAL = {"bf16": 2250.0, "e4m3": 4500.0, "mxfp4": 13500.0, "w4a8": 2250.0, "hbm": 7900.0,
           "alu": FP32_ALU_TFLOPS}
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_BYTES = 320 << 20
L2_BYTES = 129 * 10**6
KERNEL_OF = {"fp32_128": "ffma_dense_kernel", "bf16_1024": "tc_bf16_kernel",
             "bf16_4096": "tc2_gemm_kernel", "skinny_16x28672x8192": "skinny_tc_kernel",
             "mxfp4_8192": "mxfp4_pair_kernel", "e4m3_8192_bias_gelu": "tc2_gemm_kernel",
             "bf16_4096_bias_silu": "tc2_gemm_kernel", "bf16_4096_a_mn_major": "tc2_gemm_kernel", "bf16_4096_b_kn": "tc2_gemm_kernel",
             "w4a8_8192": "tc2_gemm_kernel", "w4a8_16x28672x8192": "w4a8_skinny_kernel"}


# kernel that a forced path runs (bench.py --path)
PATH_KERNEL = {"ffma": "ffma_dense_kernel", "skinny_ffma": "skinny_ffma_kernel", "skinny": "skinny_tc_kernel",
               "tc_single": "tc_bf16_kernel", "tc_pair": "tc2_gemm_kernel"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def load_traffic():
    """Per-launch DRAM bytes from committed ncu summaries, keyed by workload;
    dropped when the kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except Exception:
        return {}
    from tiled_mma_atom_gb300 import build as tb
    out = {}
    for wl, r in rec.items():
        if r.get("source_hash") == tb.source_hash(r.get("source", "")):
            out[wl] = r.get("dram_bytes_per_launch")
    return out


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workloads

def input_bytes(w):
    if w.dtype == "mxfp4":
        return (w.M + w.N) * (w.K // 2 + w.K // 32)
    if w.dtype == "w4a8":
        return w.M * w.K + w.N * w.K // 2
    elem = {"f32": 4, "bf16": 2, "e4m3": 1}[w.dtype]
    return (w.M + w.N) * w.K * elem


def l2_policy(w):
    """Flush L2 before each timed step unless the inputs alone are more than
    twice the L2 (then every step streams them from HBM anyway, and a flush
    write would only add dirty-line write-back to the timed kernel)."""
    if input_bytes(w) > 2 * L2_BYTES:
        return False, f"no flush: inputs ({input_bytes(w) / 1e6:.0f} MB) exceed twice the 129 MB L2"
    return True, (f"flushed before every timed step: {L2_FLUSH_BYTES >> 20} MiB write, then a "
                  f"{L2_CLEAN_BYTES >> 20} MiB read so the written lines are written back before the step")


class L2Flush:
    """Write a buffer larger than L2, then read another one, outside the
    timed interval: afterwards L2 holds only clean lines of the read buffer."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.zeros(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink[0])


def preshuffled_inputs(w, dev, host):
    """W4A8 workloads that take their weights pre-shuffled: the image is made
    once, on the device, before anything is timed (weights are prepared
    when they are loaded, not per call)."""
    import tiled_mma_atom_gb300 as tmg
    return [host[0], tmg.w4a8_preshuffle(host[1].to(dev)).cpu()]


def device_inputs(w, dev):
    from tiled_mma_atom_gb300 import inputs
    host = inputs.make_inputs(w)
    if w.b_preshuffled:
        host = preshuffled_inputs(w, dev, host)
    return host, [t.to(dev) for t in host]


def accumulate_note(w):
    if w.dtype != "w4a8":
        return "fp32"
    if w.M <= 64:
        return ("exact integer: offset-binary E4M3 weights on the fp8 tensor cores, fp32 column sums "
                "below 2^22, int32 epilogue")
    return "exact integer: fp32 within K segments of 8192, int32 across them"


def make_call(w, dev_in, out, stream, path="auto"):
    import tiled_mma_atom_gb300 as tmg
    if w.dtype == "mxfp4":
        A, B, sA, sB = dev_in
        return lambda: tmg.gemm_mxfp4(A, B, sA, sB, out, stream=stream)
    if w.dtype == "w4a8" and w.b_preshuffled:
        A, Bs = dev_in                    # Bs: the pre-shuffled image (see preshuffled_inputs)
        return lambda: tmg.gemm_w4a8_preshuffled(A, Bs, w.N, out, stream=stream)
    if w.dtype == "w4a8":
        A, B = dev_in
        return lambda: tmg.gemm_w4a8(A, B, out, stream=stream)
    if w.epilogue is not None:
        A, B, sa, sb, bias = dev_in
        return lambda: tmg.gemm_fused(A, B, out, scale_a=sa, scale_b=sb, bias=bias,
                                      epilogue=w.epilogue, stream=stream)
    A, B = dev_in
    if path != "auto":
        return lambda: tmg.gemm(A, B, out, path=path, stream=stream)
    if w.a_mn_major or w.b_mn_major:
        la = ((w.M, w.K), (1, w.M)) if w.a_mn_major else None
        lb = ((w.N, w.K), (1, w.N)) if w.b_mn_major else None
        return lambda: tmg.gemm(A, B, out, M=w.M, N=w.N, K=w.K, layoutA=la, layoutB=lb, stream=stream)
    return lambda: tmg.gemm(A, B, out, stream=stream)


def roofline(w, ms_per_launch, peaks, peak_kind, traffic):
    t = ms_per_launch * 1e-3
    if w.name.startswith("skinny") or (w.dtype == "w4a8" and w.M <= 64):
        if w.dtype == "w4a8":    # int8 A, 4-bit B, int32 D
            alg = w.M * w.K + w.N * w.K // 2 + w.M * w.N * 4
        else:
            alg = (w.M * w.K + w.N * w.K + w.M * w.N) * 2
        ach = alg / t / 1e9
        peak = peaks["hbm_gbs"]
        r = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
             "algorithmic_bytes": alg}
    elif w.dtype == "f32":
        ach = w.flops / t / 1e12
        peak = FP32_ALU_TFLOPS
        r = {"bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
             "peak_source": "152 SMs x 128 FP32 FMA/clk x 2 x 2.07 GHz"}
    else:
        ach = w.flops / t / 1e12
        peak = peaks["bf16_tflops"]
        src = f"{peak_kind} bf16 burst"
        if w.dtype == "mxfp4":
            peak = peak * FP4_OVER_BF16
            src = f"{peak_kind} bf16 burst x nominal fp4/bf16 ratio 6"
        elif w.dtype == "e4m3":
            peak = peak * FP8_OVER_BF16
            src = f"{peak_kind} bf16 burst x nominal fp8/bf16 ratio 2"
        if w.dtype == "w4a8":
            src = f"{peak_kind} bf16 burst (the integer products run on the bf16 tensor cores)"
        r = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
             "peak_source": src}
    r["frac"] = r["achieved"] / r["peak"]
    nominal = NOMINAL[w.dtype if r["bound"] == "tensor" else r["bound"]]
    r["nominal_peak"] = nominal
    r["frac_nominal"] = r["achieved"] / nominal
    r["traffic"] = traffic.get(w.name)
    r["kernel"] = KERNEL_OF[w.name]
    return r


def time_device(w, steps, warmup, dev, stream, flush, path="auto"):
    """Per-step CUDA-event time of one library call (inputs in HBM); `path`
    forces a kernel family for dense f32/bf16 workloads (tmg_gemm_ex)."""
    import torch
    import tiled_mma_atom_gb300 as tmg
    host, dev_in = device_inputs(w, dev)
    dt = {"f32": torch.float32, "w4a8": torch.int32}.get(w.dtype, torch.bfloat16)
    out = torch.empty((w.M, w.N), dtype=dt, device=dev)
    call = make_call(w, dev_in, out, stream, path)
    do_flush, _ = l2_policy(w)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            if do_flush:
                flush()
            call()
    tmg.check(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    n0 = tmg.launch_count()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(steps):
            if do_flush:
                flush()
            starts[i].record(stream)
            call()
            ends[i].record(stream)
    torch.cuda.synchronize()
    launches = tmg.launch_count() - n0
    tmg.check(stream)
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return ms, launches, host, dev_in, out


def time_warm(w, dev_in, out, stream, calls=20, path="auto"):
    """Mean CUDA-event time per call over `calls` back-to-back library calls
    with no flush between them (operands warm in L2 where they fit).  A spin
    kernel queued first keeps the GPU busy while the host queues the calls,
    so host submission does not pace them."""
    import torch
    import tiled_mma_atom_gb300 as tmg
    call = make_call(w, dev_in, out, stream, path)
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(4_000_000)
        s.record(stream)
        for _ in range(calls):
            call()
        e.record(stream)
    torch.cuda.synchronize()
    tmg.check(stream)
    return s.elapsed_time(e) / calls


def time_e2e(w, steps, dev, stream):
    """Same metric through the public API with host buffers: H2D of the
    inputs from pinned memory, the GEMM, D2H of D — all inside the timing.
    Dense row-major f32/bf16 workloads use the library's host-buffer call
    (tmg_gemm_host, which overlaps the transfers with the GEMM); the others
    copy with torch around the device call."""
    import torch
    import tiled_mma_atom_gb300 as tmg
    from tiled_mma_atom_gb300 import inputs
    host = inputs.make_inputs(w)
    if w.b_preshuffled:
        host = preshuffled_inputs(w, dev, host)
    host = [t.pin_memory() for t in host]
    dt = {"f32": torch.float32, "w4a8": torch.int32}.get(w.dtype, torch.bfloat16)
    out_host = torch.empty((w.M, w.N), dtype=dt).pin_memory()
    if w.dtype in ("f32", "bf16") and w.epilogue is None and not w.a_mn_major and not w.b_mn_major:
        def step():
            tmg.gemm_host(host[0], host[1], out_host, stream=stream)
    else:
        dev_in = [torch.empty_like(t, device=dev) for t in host]
        out = torch.empty((w.M, w.N), dtype=dt, device=dev)
        call = make_call(w, dev_in, out, stream)

        def step():
            for h, d in zip(host, dev_in):
                d.copy_(h, non_blocking=True)
            call()
            out_host.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(steps):
            step()
    stream.synchronize()
    dt_s = (time.perf_counter() - t0) / steps
    tmg.check(stream)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = out_host.numel() * out_host.element_size()
    return dt_s, h2d, d2h


def unit_value(w, seconds):
    return w.flops / seconds / 1e12     # TFLOP/s


def sig(x, n=4):
    """x rounded to n significant digits (keeps the JSON line short)."""
    if x is None or x == 0:
        return x
    from math import floor, log10
    return round(x, max(0, n - 1 - int(floor(log10(abs(x))))))


def config_entry(w, ms_list, rl, cpu, ms_warm=None):
    """One compact entry of the per-configuration block: GPU mean time per
    call with L2 flushed (the throughput and roofline fraction use it; the
    median is beside it), the back-to-back time with operands warm, plus the
    oracle's own timing."""
    mean = statistics.mean(ms_list)
    e = {"tflops": sig(unit_value(w, mean * 1e-3)), "ms": sig(mean), "ms_median": sig(statistics.median(ms_list)),
         **({"ms_warm": sig(ms_warm)} if ms_warm is not None else {}),
         "bound": rl["bound"],
         "achieved": sig(rl["achieved"]), "unit": rl["unit"], "frac": sig(rl["frac"], 3),
         "kernel": rl["kernel"]}
    if cpu is not None:
        v, secs, rows, thr = cpu
        e["cpu"] = {"tflops": sig(v, 3), "s": sig(secs, 3), "rows": f"{rows}/{w.M}", "cores": thr}
    return e


# ------------------------------------------------------------ CPU oracle

def oracle_sample(w, budget_s):
    """Time the fp64 oracle on the first r rows of D, r chosen so the run
    takes about budget_s.  Returns (TFLOP/s, seconds, rows, threads)."""
    import numpy as np
    import oracle
    from tiled_mma_atom_gb300 import inputs
    host = inputs.make_inputs(w)
    threads = oracle.max_threads()

    def run(rows):
        if w.dtype == "mxfp4":
            A, B, sA, sB = [t.numpy() for t in host]
            t0 = time.perf_counter()
            oracle.gemm_mxfp4(A[:rows], B, sA[:rows], sB, rows, w.N, w.K)
            return time.perf_counter() - t0
        if w.dtype == "w4a8":
            A, B = [t.numpy() for t in host]
            t0 = time.perf_counter()
            oracle.gemm_w4a8(A[:rows], B, rows, w.N, w.K)
            return time.perf_counter() - t0
        if w.epilogue is not None:
            A, B, sa, sb, bias = host
            dtype = oracle.E4M3 if w.dtype == "e4m3" else oracle.BF16
            a = inputs.bits_of(A[:rows])
            b = inputs.bits_of(B)
            t0 = time.perf_counter()
            oracle.gemm_fused(a, b, dtype, rows, w.N, w.K, sa[:rows].numpy(), sb.numpy(), bias.numpy(),
                              w.epilogue)
            return time.perf_counter() - t0
        A, B = host
        dtype = oracle.F32 if w.dtype == "f32" else oracle.BF16
        b = inputs.bits_of(B)
        lb = oracle.make_layout((w.N, w.K), (1, w.N)) if w.b_mn_major else oracle.row_major(w.N, w.K)
        if w.a_mn_major:            # the first rows of A are the first columns of its buffer
            a, la = inputs.bits_of(A), oracle.make_layout((rows, w.K), (1, w.M))
        else:
            a, la = inputs.bits_of(A[:rows]), oracle.row_major(rows, w.K)
        t0 = time.perf_counter()
        oracle.gemm(a, la, b, lb, dtype, rows, w.N, w.K)
        return time.perf_counter() - t0

    probe_rows = min(w.M, max(1, threads))
    t = run(probe_rows)
    rows = probe_rows
    if t < budget_s and rows < w.M:
        rows = int(min(w.M, max(probe_rows, probe_rows * budget_s / max(t, 1e-6))))
        t = run(rows)
    flops = 2.0 * rows * w.N * w.K
    return flops / t / 1e12, t, rows, threads


# ------------------------------------------------------------------- main

def dist_setup(n):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world, flops_per_step, steps, slowest_rank_ms):
    """Whole-job throughput: every rank ran `steps` replicas of the workload;
    the job took as long as its slowest rank."""
    return world * flops_per_step * steps / (slowest_rank_ms * 1e-3) / 1e12


def run_reference(args, world, rank, pg):
    from tiled_mma_atom_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    if rank != 0:
        return
    per_step = max(0.3, 90.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, per_step)
    vals, secs, rows, thr = [], [], 0, 0
    t_all = time.perf_counter()
    for _ in range(args.steps):
        v, s, rows, thr = oracle_sample(w, per_step)
        vals.append(v)
        secs.append(s)
    total = time.perf_counter() - t_all
    value = statistics.median(vals)
    sample = f"first {rows} of {w.M} rows of D ({rows}x{w.N}x{w.K}), fp64 oracle, median of {args.steps}"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": total}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--path", default="auto",
                    help="kernel family for a dense f32/bf16 workload (auto, ffma, tc, skinny, skinny_ffma, "
                         "tc_single, tc_pair): profiling aid, with --no-extra")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world, rank, local, pg = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank, pg)
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    import tiled_mma_atom_gb300 as tmg
    from tiled_mma_atom_gb300 import inputs

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        flush = L2Flush(dev)
    stream.synchronize()
    peaks, peak_kind = load_peaks()
    traffic = load_traffic()
    w = inputs.WORKLOADS[args.workload]

    # ---- timed region (headline) ----
    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    barrier(pg)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.05)
    t_wall = time.perf_counter()
    ms, launches, host, dev_in, out = time_device(w, args.steps, args.warmup, dev, stream, flush, args.path)
    wall = time.perf_counter() - t_wall
    torch.cuda.synchronize()
    barrier(pg)
    clk = clocks.stop()
    kernel_ms = sum(ms)
    kernel_ms_max = max_over_ranks(pg, kernel_ms)
    ms_per_step = kernel_ms_max / args.steps
    value = aggregate_tflops(world, w.flops, args.steps, kernel_ms_max)
    rl = roofline(w, kernel_ms / args.steps, peaks, peak_kind, traffic)
    if args.path != "auto":
        rl["kernel"] = PATH_KERNEL.get(args.path, args.path)
        rl["traffic"] = None

    e2e_s, h2d, d2h = time_e2e(w, max(3, min(20, args.steps)), dev, stream)
    e2e_s = max_over_ranks(pg, e2e_s)

    # the other workloads: the "next" rows first (compact), then the five
    # configurations, each with the oracle timed on the host cores; the
    # per-configuration block is the last key of the line
    cpu, cpu_head = None, None
    if rank == 0 and world == 1:
        cpu_head = oracle_sample(w, args.cpu_budget)
        v, secs, rows, thr = cpu_head
        cpu = {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"first {rows} of {w.M} rows of D ({rows}x{w.N}x{w.K}) in {secs:.1f} s, fp64"}

    extra, configs = {}, {}
    if not args.no_extra:
        for name, ow in inputs.WORKLOADS.items():
            if name == w.name or name in CONFIGS:
                continue
            try:
                steps = 400 if ow.flops < 1e11 else 100
                oms, ol, _, _, _ = time_device(ow, steps, 5, dev, stream, flush)
                per = statistics.mean(oms)
                orl = roofline(ow, per, peaks, peak_kind, traffic)
                extra[name] = {"tflops": sig(unit_value(ow, per * 1e-3)), "ms_median": sig(statistics.median(oms)),
                               "launches_per_step": ol / steps, "flushed": l2_policy(ow)[0],
                               "roofline": {k: sig(v) if isinstance(v, float) else v for k, v in orl.items()
                                            if k not in ("peak_source", "nominal_peak")}}
            except Exception as e:  # report, do not hide
                extra[name] = {"unavailable": f"{type(e).__name__}: {e}"}
        for i, name in enumerate(CONFIGS):
            ow = inputs.WORKLOADS[name]
            key = f"C{i + 1}_{name}"
            try:
                if name == w.name:
                    oms, orl = ms, rl
                    warm = time_warm(w, dev_in, out, stream, path=args.path)
                else:
                    steps = 400 if ow.flops < 1e11 else 100
                    oms, _, _, o_in, o_out = time_device(ow, steps, 5, dev, stream, flush)
                    orl = roofline(ow, statistics.mean(oms), peaks, peak_kind, traffic)
                    warm = time_warm(ow, o_in, o_out, stream)
                    del o_in, o_out
                cpu_c = None
                if rank == 0 and world == 1:
                    cpu_c = cpu_head if name == w.name else oracle_sample(ow, CONFIG_CPU_BUDGET)
                configs[key] = config_entry(ow, oms, orl, cpu_c, warm)
            except Exception as e:  # report, do not hide
                configs[key] = {"unavailable": f"{type(e).__name__}: {e}"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                       "a": w.a_dist, "b": w.b_dist,
                       "accumulate": accumulate_note(w),
                       **({"epilogue": w.epilogue} if w.epilogue else {}),
                       "l2": l2_policy(w)[1],
                       "timing": "CUDA events around each library call on its stream",
                       **({"path": args.path} if args.path != "auto" else {}),
                       "ms_median": statistics.median(ms), "ms_min": min(ms),
                       "parallelism": f"{world} independent replica(s)"},
            "roofline": rl,
            "cpu_baseline": cpu,
            "e2e": {"value": unit_value(w, e2e_s) * world, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": int(launches),
            "clocks": clk,
            "peaks": {"source": peak_kind, **peaks},
            "timed_wall_s": wall,
            "workloads": extra,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
