#!/usr/bin/env python
"""Benchmark of the dense tiled GEMM on GB300.

One step = one GEMM call (the whole hot path) on the 4096 x 4096 x 8192
FP16-in / FP16-out workload (FP32 accumulation), the compute-bound shape of
"Two Waves, One Stage Apart" (section "MI350 Series"). Throughput is
2*M*N*K / elapsed, as in that page's Table 1 caption.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed warm-up steps, then exactly K steps between a barrier and
torch.cuda.synchronize() on both sides. CUDA events are recorded on the
launching stream at both ends of the timed region; the mean launch duration
is the region time over K. Operands rotate over enough
(A, B, C) sets to exceed twice the L2 size, so every step reads from HBM.
The SM clock of each timed launch is measured inside the kernel (the clock
trace option: CTA 0's cycle counter over the global timer), and nvidia-smi
is sampled during the timed region for throttle reasons; its clock counts
only from samples that drew load power.
Under torchrun (N > 1) every rank runs its own replica; the time is the
maximum over ranks, and rank 0 prints one JSON line.

--impl reference times the CPU FP64 oracle on this host instead, on a
bounded sample of rows of the same workload per step.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "GEMM TFLOP/s at 4096x4096x8192 FP16 and % of GB300 dense tensor peak"
PAGES_REFERENCE_TFLOPS = 1437.0   # MI355X, 8-wave warp-pipelined Triton, same shape (context only)
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_DENSE_TFLOPS = 2250.0     # GB300 dense FP16/BF16 tensor peak, nominal
FP8_RATE = 2.0                    # nominal dense FP8 / FP16 rate on GB300 (4.5 vs 2.25 PFLOP/s)
FP4_RATE = 6.0                    # nominal dense FP4 / FP16 rate on GB300 (13.5 vs 2.25 PFLOP/s)
# Dense tensor flop per SM clock, measured with back-to-back tcgen05.mma products:
# FP16/BF16 8,192; FP8 and MXFP8 twice that; every packed-FP4 form four times.
FLOP_PER_SM_CLOCK = {1.0: 8192.0, FP8_RATE: 16384.0, FP4_RATE: 32768.0}


def clock_peak_tflops(rate: float, sms: int, sm_mhz: float) -> float:
    """Tensor peak at the sampled SM clock: SMs x measured flop per SM clock x clock."""
    return sms * FLOP_PER_SM_CLOCK[rate] * sm_mhz * 1e6 / 1e12


def is_mx(w) -> bool:
    return w.dtype_in in workloads.MX_ELEMENT


def rate_of(w) -> float:
    """Nominal dense tensor rate of the workload's input type, relative to FP16/BF16."""
    elem = workloads.MX_ELEMENT.get(w.dtype_in, w.dtype_in)
    return FP4_RATE if elem == "e2m1" else FP8_RATE if elem in workloads.FP8 else 1.0


def oracle_operands(w):
    """The workload's operands as the oracle takes them (raw patterns, and scales for MX)."""
    ops = workloads.workload_operands(w)
    return tuple(workloads.as_bits(t) for t in ops)


def oracle_rows(oracle, w, ops, rows, threads):
    if is_mx(w):
        A, B, SFA, SFB = ops
        return oracle.gemm_ref_mx(A, B, SFA, SFB, w.M, w.N, w.K, workloads.MX_ELEMENT[w.dtype_in],
                                  rows=rows, threads=threads)
    A, B = ops
    return oracle.gemm_ref(A, B, w.M, w.N, w.K, w.dtype_in, w.layout_b, rows=rows, threads=threads)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.HEADLINE,
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.ATTENTION_WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--compare-cublas", action="store_true",
                    help="also time torch.matmul (cuBLAS) the same way, as a labelled comparison")
    ap.add_argument("--stream-k", choices=["auto", "off", "on"], default="auto",
                    help="tail scheduling of the GEMM (gemm_options_t.stream_k); auto = the planner")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--graph", action="store_true",
                    help="capture the timed steps into one CUDA graph and time its replay "
                         "(no per-launch host cost; GEMM workloads)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    return ap.parse_args()


# ---------------------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# The files each kernel and its launcher are built from; a profile summary
# names this hash, and its DRAM traffic is reported only while it matches.
GEMM_SOURCES = ("gemm.cu", "gemm_kernel.cuh", "ptx.cuh", "schedule.cuh", "runtime.h")
ATTENTION_SOURCES = GEMM_SOURCES + ("attention.cu", "attention_kernel.cuh")


def source_hash(sources=GEMM_SOURCES) -> str:
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "dense_tiled_gemm_gb300", "csrc", name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def max_over_ranks(x: float, pg, device) -> float:
    """Maximum of a per-rank scalar over all ranks (identity without a process group)."""
    if pg is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, seconds: float) -> float:
    """Units all ranks processed divided by the slowest rank's time."""
    return world * flops_per_step * steps / seconds / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return json.load(fh), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": 6800.0}, "fallback"


def profiled_traffic(workload: str, sources=GEMM_SOURCES):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it is now; otherwise None."""
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        with open(path) as fh:
            text = fh.read()
        wl = re.search(r"^workload:\s*(\S+)", text, re.M)
        src = re.search(r"^source_sha256:\s*(\S+)", text, re.M)
        tr = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        if wl and src and tr and wl.group(1) == workload and src.group(1) == source_hash(sources):
            return float(tr.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as fh:
            lines = [ln.strip() for ln in fh if ln.strip()]
        os.unlink(self.tmp.name)
        sm, sm_max, power, reasons = [], 0.0, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                sm_max = max(sm_max, float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        # only samples taken while the GPU drew load power count; a region shorter
        # than the sampling period may have none, and then no clock is claimed
        loaded = [s for s, p in zip(sm, power) if p > 300.0]
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": sm_max,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(loaded),
                "power_w_max": max(power) if power else None}


# %globaltimer advances in steps, not every nanosecond: a launch of a few
# microseconds can read a quarter above the maximum clock from one interval.
# Below SHORT_LAUNCH_NS of median launch length the clock is pooled over all
# launches; below TOO_SHORT_NS even that read 35% above the maximum clock
# (256^3, ~3 us launches), so no in-kernel clock is reported.
SHORT_LAUNCH_NS = 20000
TOO_SHORT_NS = 5000


def kernel_clock_mhz(trace: torch.Tensor) -> dict:
    """SM clock of the traced launches from their clock_trace words (global timer ns
    and SM cycles of CTA 0 at its start and end), in MHz: per launch (cycles / ns), and
    pooled over all launches (all cycles / all ns), which averages out the timer's steps."""
    t = trace.cpu().tolist()
    spans = [(n1 - n0, c1 - c0) for n0, c0, n1, c1 in t if n1 > n0 and c1 > c0]
    if not spans:
        return {"per_launch": [], "pooled": None, "median_ns": None}
    return {"per_launch": [c / n * 1e3 for n, c in spans],
            "pooled": sum(c for _, c in spans) / sum(n for n, _ in spans) * 1e3,
            "median_ns": statistics.median(n for n, _ in spans)}


def merge_clocks(smi: dict | None, kc: dict | None) -> dict | None:
    """The line's clock record: the in-kernel SM clock where the launches were traced
    (the median over the timed launches, or for launches shorter than SHORT_LAUNCH_NS
    the pooled clock), nvidia-smi's samples under load otherwise; throttle reasons and
    the maximum clock always come from nvidia-smi."""
    out = dict(smi) if smi else {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                                 "samples_under_load": 0, "power_w_max": None}
    out["smi_sm_mhz_under_load"] = out.get("sm_mhz")
    mhz = kc["per_launch"] if kc else []
    max_mhz = out.get("sm_max_mhz")
    pooled_ok = bool(mhz) and (max_mhz is None or kc["pooled"] <= 1.02 * max_mhz)
    if mhz and (kc["median_ns"] < TOO_SHORT_NS or not pooled_ok):
        out["kernel_mhz_min"] = min(mhz)
        out["kernel_mhz_max"] = max(mhz)
        out["sm_mhz_source"] = (f"in-kernel clock not used: median launch {kc['median_ns'] / 1e3:.1f} us, too short "
                                "for the global timer's steps; " +
                                ("nvidia-smi samples drawing > 300 W" if out.get("sm_mhz") is not None
                                 else "no nvidia-smi sample under load"))
        mhz = []
        return out
    if mhz:
        n = len(mhz)
        if kc["median_ns"] < SHORT_LAUNCH_NS:
            out["sm_mhz"] = kc["pooled"]
            out["sm_mhz_source"] = (f"in-kernel: SM cycles over global-timer ns of CTA 0, pooled over {n} "
                                    f"timed launches (median launch {kc['median_ns'] / 1e3:.1f} us, too short "
                                    "for the timer's steps)")
        else:
            out["sm_mhz"] = statistics.median(mhz)
            out["sm_mhz_source"] = (f"in-kernel: SM cycles over global-timer ns of CTA 0, median of {n} "
                                    "timed launches")
        out["kernel_mhz_min"] = min(mhz)
        out["kernel_mhz_max"] = max(mhz)
    else:
        out["sm_mhz_source"] = ("nvidia-smi samples drawing > 300 W" if out.get("sm_mhz") is not None
                                else "none: no sample under load")
    return out


def oracle_sample(w, ops, rows_total: int, threads: int):
    """Time the oracle on `rows_total` output rows of workload w (FP64, host cores)."""
    import oracle
    rows = list(range(0, w.M, max(1, w.M // rows_total)))[:rows_total]
    t0 = time.perf_counter()
    oracle_rows(oracle, w, ops, rows, threads)
    return time.perf_counter() - t0, len(rows)


def cpu_baseline(w, target_s: float) -> dict:
    import oracle
    threads = oracle.host_threads()
    ops = oracle_operands(w)
    t1, r1 = oracle_sample(w, ops, threads, threads)       # one row per thread: calibration
    rows = max(threads, min(w.M, int(r1 * target_s / max(t1, 1e-3))))
    rows = max(threads, rows // threads * threads)
    t, r = oracle_sample(w, ops, rows, threads)
    flops = 2.0 * r * w.N * w.K
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{r} of {w.M} output rows (all {w.N} columns, K={w.K}), FP64 i-k-j loop, "
                      f"{t:.1f} s wall including the FP64 decode of B",
            "seconds": t}


# ---------------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = workloads.WORKLOADS[args.workload]
    threads = oracle.host_threads()
    ops = oracle_operands(w)
    # Each oracle call decodes B once (a fixed cost) and then computes its rows,
    # one per thread at a time. Calibrate both: one call with a single row (the
    # fixed cost and one row time), one with two rows per thread (one more row
    # time), so a row costs (difference) / threads at full width.
    t0 = time.perf_counter()
    oracle_rows(oracle, w, ops, [0], threads)
    t_one = time.perf_counter() - t0
    n_cal = min(2 * threads, w.M)
    t0 = time.perf_counter()
    oracle_rows(oracle, w, ops, list(range(n_cal)), threads)
    t_row = max((time.perf_counter() - t0 - t_one) / threads, 1e-6)
    # every timed step takes the same number of rows; the whole timed run is one
    # oracle call over all steps' rows (so B is decoded once), sized to ~60 s
    budget = 60.0
    rows = max(1, min(4 * threads, w.M, int(max(budget - t_one, 1.0) / t_row / max(1, args.steps))))
    stride = max(1, w.M // rows)
    samples = [list(range((s * 7) % stride, w.M, stride))[:rows] for s in range(args.steps + args.warmup)]
    for s in range(min(args.warmup, 2)):
        oracle_rows(oracle, w, ops, samples[s], threads)
    timed_rows = [r for s in range(args.steps) for r in samples[args.warmup + s]]
    rows = len(timed_rows) // max(1, args.steps)
    t0 = time.perf_counter()
    oracle_rows(oracle, w, ops, timed_rows, threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * len(timed_rows) * w.N * w.K
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGES_REFERENCE_TFLOPS if w.name == workloads.HEADLINE else None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype_in": w.dtype_in,
                   "dtype_out": w.dtype_out, "layout_b": w.layout_b,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} of {w.M} output rows per step, all {w.N} columns; the "
                                   f"{args.steps} steps' rows in one oracle call (one decode of B)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def time_cublas(As, Bs, Cs, w, n_sets, args, stream, smi_id, pg, dev) -> dict:
    """torch.matmul (cuBLAS) on the same rotating operands, timed the same way.
    A comparison only: nothing on the product path calls it."""
    same_dtype = Cs[0].dtype == As[0].dtype
    fp8 = w.dtype_in in workloads.FP8
    how = "torch.matmul (cuBLAS)"
    if fp8:
        one = torch.ones((), dtype=torch.float32, device=dev)
        how = f"torch._scaled_mm unit scales, out_dtype={Cs[0].dtype} (cuBLASLt FP8)"
    elif not same_dtype:
        try:   # cuBLAS writing the wider output type directly, where this torch has it
            torch.mm(As[0], Bs[0].t() if w.layout_b == "k" else Bs[0], out_dtype=Cs[0].dtype)
            how = f"torch.mm out_dtype={Cs[0].dtype} (cuBLAS)"
        except (TypeError, RuntimeError):
            how = f"torch.matmul (cuBLAS), output in {As[0].dtype}: no FP32-output path in this torch"

    def step(i):
        j = i % n_sets
        Bj = Bs[j].t() if w.layout_b == "k" else Bs[j]
        if fp8:
            torch._scaled_mm(As[j], Bj, scale_a=one, scale_b=one, out_dtype=Cs[j].dtype)
        elif same_dtype:
            torch.matmul(As[j], Bj, out=Cs[j])
        elif how.startswith("torch.mm"):
            torch.mm(As[j], Bj, out_dtype=Cs[j].dtype)
        else:
            torch.matmul(As[j], Bj)
    for i in range(args.warmup):
        step(i)
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(smi_id)
    sampler.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    ev_start.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    region_ms = max_over_ranks(ev_start.elapsed_time(ev_end), pg, dev)
    kernel_ms = region_ms / args.steps
    return {"impl": how, "value": w.flops * args.steps / (region_ms * 1e-3) / 1e12,
            "unit": "TFLOP/s", "kernel_ms": kernel_ms, "clocks": clocks}


# ---------------------------------------------------------------------------- our arm
def run_ours(args):
    world, rank, local = dist_env()
    import dense_tiled_gemm_gb300 as dtg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    w = workloads.WORKLOADS[args.workload]
    out_dt = workloads.DTYPES[w.dtype_out]
    ops0 = workloads.workload_operands(w)     # (A, B) or, block-scaled, (A, B, SFA, SFB)
    A0, B0 = ops0[0], ops0[1]
    in_bytes = A0.element_size()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = sum(t.numel() * t.element_size() for t in ops0) + w.M * w.N * torch.finfo(out_dt).bits // 8
    n_sets = max(2, math.ceil(2 * l2 / set_bytes) + 1)

    def rolled(t, i):
        # rotate rows through a same-width integer view (no roll kernel for FP8 types)
        bits_dt = torch.uint8 if t.element_size() == 1 else torch.int16
        return t.to(dev) if i == 0 else t.to(dev).view(bits_dt).roll(i, 0).view(t.dtype)

    sets, Cs = [], []
    for i in range(n_sets):
        sets.append([rolled(t, i) for t in ops0])
        Cs.append(torch.empty((w.M, w.N), dtype=out_dt, device=dev))
    As, Bs = [st[0] for st in sets], [st[1] for st in sets]
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)

    opts = None if args.stream_k == "auto" else {"stream_k": {"off": 1, "on": 2}[args.stream_k]}
    # each timed launch writes its own clock-trace words (CTA 0's global timer and SM
    # cycle counter at its start and end): the clock the kernel ran at
    trace = torch.zeros((args.steps, 4), dtype=torch.int64, device=dev)
    timed_opts = []
    for i in range(args.steps):
        o = dtg.GemmOptions()
        if opts:
            o.stream_k = opts["stream_k"]
        o.clock_trace = trace[i].data_ptr()
        timed_opts.append(o)

    def step(i, st=stream, o=opts):
        j = i % n_sets
        if is_mx(w):
            A, B, SFA, SFB = sets[j]
            dtg.gemm_mx(A, B, SFA, SFB, Cs[j], K=w.K, stream=st, options=o)
        else:
            dtg.gemm(As[j], Bs[j], Cs[j], layout_b=w.layout_b, stream=st, options=o)

    for i in range(args.warmup):
        step(i)
    status, detail = dtg.gemm_last_device_status(stream)
    if status != dtg.GEMM_OK:
        raise RuntimeError(f"device status {dtg.gemm_status_string(status)} site {detail:#x}")

    # Events only at the two ends of the timed region: an event recorded between
    # two launches would stop the next launch from overlapping the previous one.
    # Only this kernel runs on the stream here, so the mean launch duration is
    # the region time over the step count.
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    try:
        smi_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001  (older torch: fall back to the CUDA index)
        smi_id = str(local)
    graph = None
    if args.graph:
        # the same steps, captured once (launches are counted at capture) and replayed
        # once untimed; the timed region is then one replay on this stream
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(dev)
        launches0 = dtg.gemm_launch_count()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                step(args.warmup + i, st=None, o=timed_opts[i])
        launches = dtg.gemm_launch_count() - launches0
        graph.replay()
        torch.cuda.synchronize(dev)
    sampler = ClockSampler(smi_id)
    sampler.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    if graph is None:
        launches0 = dtg.gemm_launch_count()
    ev_start.record(stream)
    if graph is None:
        for i in range(args.steps):
            step(args.warmup + i, o=timed_opts[i])
    else:
        graph.replay()
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    if graph is None:
        launches = dtg.gemm_launch_count() - launches0
    clocks = merge_clocks(sampler.stop(), kernel_clock_mhz(trace))
    status, detail = dtg.gemm_last_device_status(stream)
    if status != dtg.GEMM_OK:
        raise RuntimeError(f"device status {dtg.gemm_status_string(status)} site {detail:#x}")

    region_ms = ev_start.elapsed_time(ev_end)
    kernel_ms = region_ms / args.steps
    region_ms = max_over_ranks(region_ms, pg, dev)
    flops_step = float(w.flops)
    value = whole_job_tflops(world, flops_step, args.steps, region_ms * 1e-3)

    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))  # FP16 and BF16 share the dense rate
    rate = rate_of(w)
    nominal = NOMINAL_DENSE_TFLOPS * rate
    if rate != 1.0:
        peak *= rate
        peak_note = (f"{peak_src} bf16_tflops (burst) x {rate:g}, the nominal dense ratio of this "
                     "input type to BF16 (FP8 4.5, FP4 13.5 vs 2.25 PFLOP/s)")
    else:
        peak_note = f"{peak_src} bf16_tflops (burst); FP16 dense rate = BF16"
    achieved = flops_step / (kernel_ms * 1e-3) / 1e12
    plan = dtg.gemm_plan(w.M, w.N, w.K, dtype_in=A0.dtype, dtype_out=out_dt,
                         layout_b=w.layout_b, a_ptr=As[0].data_ptr(), b_ptr=Bs[0].data_ptr(),
                         c_ptr=Cs[0].data_ptr(), options=opts, block_scaled=is_mx(w))

    cublas = None
    if args.compare_cublas and not is_mx(w):
        cublas = time_cublas(As, Bs, Cs, w, n_sets, args, stream, smi_id, pg, dev)
    elif args.compare_cublas:
        cublas = {"impl": None, "note": "no block-scaled library GEMM is timed for comparison"}

    e2e = None
    if not args.no_e2e and not is_mx(w):
        Ah = A0.pin_memory()
        Bh = B0.pin_memory()
        Chs = [torch.empty((w.M, w.N), dtype=out_dt).pin_memory() for _ in range(2)]
        for Ch in Chs:   # grows both staging slots
            dtg.gemm_from_host_async(Ah, Bh, Ch, layout_b=w.layout_b, stream=stream)
        torch.cuda.synchronize(dev)
        n = max(1, args.e2e_steps)
        if pg:
            pg.barrier()
        # every step uploads its A and B from pinned host memory and reads its C back;
        # consecutive calls overlap one step's uploads with the previous step's product
        # and read-back, and the region ends when the last read-back has landed
        t0 = time.perf_counter()
        for i in range(n):
            dtg.gemm_from_host_async(Ah, Bh, Chs[i % 2], layout_b=w.layout_b, stream=stream)
        torch.cuda.synchronize(dev)
        dt = max_over_ranks(time.perf_counter() - t0, pg, dev)
        dtg.gemm_release_workspace()
        e2e = {"value": whole_job_tflops(world, flops_step, n, dt), "unit": "TFLOP/s",
               "h2d_bytes_per_step": (Ah.numel() + Bh.numel()) * in_bytes,
               "d2h_bytes_per_step": Chs[0].numel() * Chs[0].element_size(),
               "steps": n, "api": "gemm_from_host_async (pinned host buffers; one step's uploads overlap "
                                  "the previous step's product and read-back)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": region_ms / args.steps,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / world / PAGES_REFERENCE_TFLOPS if w.name == workloads.HEADLINE else None,
            "vs_baseline_ref": "1437 TFLOP/s: MI355X 8-wave warp-pipelined Triton, same shape (context)",
            "dtype": w.dtype_in, "accumulate": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype_in": w.dtype_in,
                       "dtype_out": w.dtype_out, "layout_b": w.layout_b,
                       "l2": f"rotating {n_sets} operand sets "
                             f"({n_sets * set_bytes / 1e6:.0f} MB > 2 x {l2 / 1e6:.0f} MB L2)",
                       "parallelism": f"replicas x{world}", "plan": plan,
                       "timing": "one CUDA graph replay of all steps" if graph is not None
                                 else "back-to-back launches"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                         "peak_source": peak_note,
                         "kernel_ms": kernel_ms},
            "clocks": clocks,
            "gpu_launches": launches,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "cublas_comparison": cublas,
        }
        line["roofline"]["frac_of_nominal"] = achieved / nominal
        if "bf16_tflops_sustained" in peaks:
            # cuBLAS in a seconds-long loop under the power cap: the figure for runs the cap reaches
            sus = float(peaks["bf16_tflops_sustained"]) * rate
            line["roofline"]["sustained_peak"] = sus
            line["roofline"]["frac_of_sustained_peak"] = achieved / sus
        if clocks and clocks.get("sm_mhz"):
            cp = clock_peak_tflops(rate, torch.cuda.get_device_properties(dev).multi_processor_count,
                                   clocks["sm_mhz"])
            line["roofline"]["clock_peak_tflops"] = cp
            line["roofline"]["frac_of_clock_peak"] = achieved / cp
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------- attention
def run_attention(args):
    """The attention forward workloads: one step = one attention_fwd call over all
    B x H heads, rotating (Q, K, V, O) sets larger than 2 x L2; FLOPs = 4 * B * H *
    (visible query-key pairs) * d, as in the two products of the forward pass."""
    world, rank, local = dist_env()
    import dense_tiled_gemm_gb300 as dtg
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    w = workloads.ATTENTION_WORKLOADS[args.workload]
    Q0, K0, V0 = workloads.make_attention_operands(w.B, w.H, w.Lq, w.Lk, w.d, w.dtype, w.dist, w.seed)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = 2 * (2 * Q0.numel() + K0.numel() + V0.numel())
    n_sets = max(2, math.ceil(2 * l2 / set_bytes) + 1)
    sets = []
    for i in range(n_sets):
        sets.append([t.to(dev).view(torch.int16).roll(i, 2).view(t.dtype) if i else t.to(dev)
                     for t in (Q0, K0, V0)] + [torch.empty_like(Q0, device=dev)])
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    def step(i):
        Q, K, V, O = sets[i % n_sets]
        dtg.attention(Q, K, V, causal=w.causal, O=O, stream=stream)

    for i in range(args.warmup):
        step(i)
    status, detail = dtg.gemm_last_device_status(stream)
    if status != dtg.GEMM_OK:
        raise RuntimeError(f"device status {dtg.gemm_status_string(status)} site {detail:#x}")
    try:
        smi_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001
        smi_id = str(local)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(smi_id)
    sampler.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    launches0 = dtg.gemm_launch_count()
    ev0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    launches = dtg.gemm_launch_count() - launches0
    clocks = sampler.stop()
    clocks = merge_clocks(clocks, None)
    status, detail = dtg.gemm_last_device_status(stream)
    if status != dtg.GEMM_OK:
        raise RuntimeError(f"device status {dtg.gemm_status_string(status)} site {detail:#x}")
    region_ms = ev0.elapsed_time(ev1)
    kernel_ms = region_ms / args.steps
    region_ms = max_over_ranks(region_ms, pg, dev)
    value = whole_job_tflops(world, float(w.flops), args.steps, region_ms * 1e-3)
    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12

    comparison = None
    if args.compare_cublas:
        # torch's fused attention (its flash / cuDNN kernels), timed the same way; a comparison only
        import torch.nn.functional as F

        def tstep(i):
            Q, K, V, _ = sets[i % n_sets]
            F.scaled_dot_product_attention(Q, K, V, is_causal=w.causal and w.Lq == w.Lk)
        for i in range(args.warmup):
            tstep(i)
        sampler = ClockSampler(smi_id)
        sampler.start()
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for i in range(args.steps):
            tstep(i)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        tclk = sampler.stop()
        t_ms = ev0.elapsed_time(ev1) / args.steps
        comparison = {"impl": "torch.nn.functional.scaled_dot_product_attention", "kernel_ms": t_ms,
                      "value": w.flops / (t_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "clocks": tclk}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        threads = oracle.host_threads()
        bits = [t.contiguous().view(torch.int16).numpy() for t in (Q0, K0, V0)]
        total = w.B * w.H * w.Lq
        n = threads * 4
        t0 = time.perf_counter()
        oracle.attention_ref(*bits, w.B, w.H, w.Lq, w.Lk, w.d, w.dtype, w.causal,
                             rows=list(range(0, total, max(1, total // n)))[:n], threads=threads)
        dt = time.perf_counter() - t0
        per_row = w.flops / total
        cpu = {"value": n * per_row / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} of {total} query rows, FP64 plain softmax(QK^T)V", "seconds": dt}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": region_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "accumulate": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "d": w.d,
                       "causal": w.causal, "flops_per_step": w.flops,
                       "l2": f"rotating {n_sets} (Q, K, V, O) sets", "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(w.name, ATTENTION_SOURCES),
                         "peak_source": f"{peak_src} bf16_tflops (burst)", "kernel_ms": kernel_ms,
                         "frac_of_nominal": achieved / NOMINAL_DENSE_TFLOPS},
            "clocks": clocks, "gpu_launches": launches, "e2e": None, "cpu_baseline": cpu,
            "library_comparison": comparison,
        }
        if "bf16_tflops_sustained" in peaks:
            sus = float(peaks["bf16_tflops_sustained"])
            line["roofline"]["sustained_peak"] = sus
            line["roofline"]["frac_of_sustained_peak"] = achieved / sus
        if clocks and clocks.get("sm_mhz"):
            cp = clock_peak_tflops(1.0, torch.cuda.get_device_properties(dev).multi_processor_count,
                                   clocks["sm_mhz"])
            line["roofline"]["clock_peak_tflops"] = cp
            line["roofline"]["frac_of_clock_peak"] = achieved / cp
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.workload in workloads.ATTENTION_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the GEMM workloads"}))
            return 0
        if args.graph:
            sys.exit("--graph times GEMM workloads only (an attention launch is not launch-bound)")
        return run_attention(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
