"""Throughput of D = alpha * op(A) @ op(B) + beta * C on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--case NAME] [--no-e2e] [--no-cpu-baseline]
                    [--no-per-config] [--no-clock-study] [--cpu-budget SECONDS]
    python bench.py --library-peaks

A step is one GEMM call through the C ABI over the resident, seeded
synthetic inputs of the workload (default: M = N = K = 8192, fp16
operands drawn N(0, 1/sqrt(K)), alpha = 1, beta = 0, fp32 D).  The timed
region is exactly K steps between CUDA events on the launching stream,
bracketed by a barrier and a device synchronisation; with N > 1 (torchrun)
every rank runs its own replica and the slowest rank's time is used.

The roofline's tensor peak is the measured cuBLAS bf16 figure (x 2 for
8-bit operands) in the power state the timed loop ran in: the sustained
figure for a loop long enough to meet the power cap, the burst figure for a
short loop and for the separate burst measurement (best of three 10-launch
runs).

At N = 1 the line also carries, outside the timed region:
  clocks       the SM clock the timed loop ran at: the same loop run again
               with the grid planned for 2 fewer SMs while a one-thread
               probe kernel (compiled by this script) samples %globaltimer
               and %clock64 on a free SM.  Neither a probe between launches
               nor NVML sees it: the power limiter lets the clock back up
               within ~0.1 ms of the load stopping, and NVML reports the
               clock the controller asks for (2070 MHz during a burst that
               runs at ~1.6-1.7 GHz);
  clock_study  the headline workload for >= 1.5 s in chunks of launches,
               clocked the same way: launch time against the SM clock it
               ran at, binned by clock;
  per_config   every BASELINE workload (10 warm-ups, then >= 50 launches
               and >= 200 ms): median and min per launch, throughput,
               bound and fraction of the measured peak, and the SM clock
               during the loop (measured as above);
  cpu_baseline the oracle as it stands on the host cores, single-threaded
               and on all cores, for every workload: the full problem for
               the small ones (and 4096^3), a tile-covering sample (one
               full row per 128-row block, one full column per 256-column
               block) for the others, with the full time extrapolated from
               the measured rate and labelled so.

--impl reference times the CPU oracle instead (the only other
implementation of this operation in the repository), on bounded samples
of the same workload, on the host cores.

--library-peaks measures, instead of this library, the vendor library's
8192^3 throughput through torch (cuBLAS bf16, cuBLASLt E4M3 with per-tensor
scales to bf16 and to fp32 D): the burst (best of three 10-launch runs after
an idle second) and the sustained rate (median of the last half of a 3 s
loop).  It gives the 8-bit peak that the tensor fractions of 8-bit
workloads can be read against; the line's own fractions keep the measured
bf16 figure x 2.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s at 1 GB300 and % of dense fp16/bf16 tensor-core peak"
UNIT = "TFLOP/s"
NOMINAL_DENSE_TFLOPS = 2250.0        # GB300 dense fp16/bf16, NVIDIA's figure
FLOP_PER_CLK_PER_SM = 8192           # dense f16/bf16 tcgen05 rate per SM
FP8_RATE = 2.0                       # nominal dense fp8 rate / fp16 rate (4.5 / 2.25 PFLOP/s)
E2E_STREAMS = 2                      # streams the end-to-end steps alternate between
BURST_STEPS = 10                     # launches per burst measurement
KERNEL_SOURCES = ["dense_tensor_core_02_gb300/csrc/gemm_tcgen05.cuh",
                  "dense_tensor_core_02_gb300/csrc/gemm_sm103.cu",
                  "dense_tensor_core_02_gb300/csrc/gemm_sm103_f8.cu",
                  "dense_tensor_core_02_gb300/csrc/gemm_sm103_mx.cu",
                  "dense_tensor_core_02_gb300/csrc/ptx.cuh",
                  "dense_tensor_core_02_gb300/csrc/gemm_params.h"]


def _rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def slowest_rank_ms(elapsed_ms, dist=None, device="cpu"):
    """The job's time: the maximum over ranks of each rank's time (every
    rank runs its own replica; the job is done when the slowest is)."""
    if dist is None:
        return elapsed_ms
    import torch
    t = torch.tensor([elapsed_ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_step, steps, elapsed_ms):
    """Whole-job throughput: the flops of all ranks' steps over the job's time."""
    return world * flops_per_step * steps / (elapsed_ms * 1e-3) / 1e12


def _measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled(case_name):
    """The committed ncu figures of a workload (profiles/traffic_<case>.txt)
    if they were taken on the current kernel source, else {}."""
    path = os.path.join(ROOT, "profiles", "traffic_%s.txt" % case_name)
    if not os.path.exists(path):
        return {}
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return {}
    return vals


def _profiled_traffic(case_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        return int(float(_profiled(case_name)["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def _profiled_duration_us(case_name):
    """The ncu launch duration (us) in the committed summary, on the current
    kernel source; else None."""
    try:
        return float(_profiled(case_name)["ncu_duration_ns"]) / 1e3
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, util_sm, reasons, power = [], [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                clk, cmax, pw, util = float(parts[1]), float(parts[2]), float(parts[3]), float(parts[4])
            except ValueError:
                continue
            sm.append(clk)
            smax.append(cmax)
            power.append(pw)
            if util >= 50:
                util_sm.append(clk)
            for name, flag in zip(names, parts[6:10]):
                if flag.lower() == "active":
                    reasons.add(name)
        pick = util_sm or sm
        return {"sm_mhz": statistics.median(pick) if pick else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(util_sm),
                "power_w_max": max(power) if power else None}


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--case", default=None, help="workload name (default: the 8192^3 fp16 headline)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-clock-study", action="store_true", help="skip the clock study")
    ap.add_argument("--clock-study-seconds", type=float, default=1.5)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=100.0,
                    help="target wall time of the whole CPU oracle table (all workloads, both thread counts)")
    ap.add_argument("--library-peaks", action="store_true",
                    help="measure the vendor library's bf16 and E4M3 8192^3 throughput instead (one JSON line)")
    return ap.parse_args()


def library_peaks():
    """cuBLAS / cuBLASLt 8192^3 throughput through torch, burst and
    sustained (see the module docstring).  Measurement only: the library's
    own path never calls them."""
    import torch

    n = 8192
    flop = 2.0 * n ** 3
    g = torch.Generator(device="cuda").manual_seed(3)
    a16 = torch.randn(n, n, device="cuda", generator=g).to(torch.bfloat16)
    b16 = torch.randn(n, n, device="cuda", generator=g).to(torch.bfloat16).t()
    a8 = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn)
    b8 = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn).t()   # column-major, as cuBLASLt wants
    one = torch.ones((), device="cuda")
    ops = {
        "bf16_to_bf16": lambda: torch.mm(a16, b16),
        "e4m3_to_bf16": lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.bfloat16),
        "e4m3_to_f32": lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.float32),
    }
    out = {"workload": "M=N=K=8192, random operands", "unit": UNIT}
    for name, fn in ops.items():
        try:
            fn()
            torch.cuda.synchronize()
        except Exception as e:   # an op this torch build or GPU does not offer
            out[name] = {"unavailable": str(e).splitlines()[0][:200]}
            continue
        burst = []
        for _ in range(3):
            time.sleep(1.0)
            e0, e1 = _event_pair(torch)
            e0.record()
            for _ in range(10):
                fn()
            e1.record()
            torch.cuda.synchronize()
            burst.append(flop * 10 / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        time.sleep(1.0)
        rates = []
        t_end = time.time() + 3.0
        while time.time() < t_end:
            e0, e1 = _event_pair(torch)
            e0.record()
            for _ in range(20):
                fn()
            e1.record()
            torch.cuda.synchronize()
            rates.append(flop * 20 / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        tail = rates[len(rates) // 2:]
        out[name] = {"burst": max(burst), "burst_runs": burst, "sustained": statistics.median(tail),
                     "sustained_chunks": len(tail)}
    for kind in ("burst", "sustained"):
        if "burst" in out.get("bf16_to_bf16", {}) and "burst" in out.get("e4m3_to_f32", {}):
            out["e4m3_to_f32_over_bf16_" + kind] = out["e4m3_to_f32"][kind] / out["bf16_to_bf16"][kind]
    print(json.dumps(out), flush=True)
    return 0


def _workload_config(case, n_gpus):
    from dense_tensor_core_02_gb300.inputs import CASES
    dist = ("uniform random E2M1 codes, packed" if case.in_dtype == "e2m1" else
            ("N(0,%g)" % case.std) if case.dist == "normal" else "U[-1,1]")
    mx = (", MX block scales (UE8M0 per 32 K, bytes U{%d..%d})" % (case.sf_lo, case.sf_hi)) if case.mx else ""
    return {
        "workload": "%s: M=%d N=%d K=%d, %s A/B %s%s, %s D, alpha=%g beta=%g, transA=%d transB=%d" % (
            case.name, case.M, case.N, case.K, case.in_dtype, dist, mx, case.out_dtype, case.alpha, case.beta,
            case.transA, case.transB),
        "M": case.M, "N": case.N, "K": case.K, "accumulate": "f32", "out_dtype": case.out_dtype,
        "seed": case.seed, "workload_index": CASES.index(case) + 1,
        "l2": "inputs larger than L2 (A+B+D = %.0f MiB > 129 MB), no flush" % (case.algorithmic_bytes / 2 ** 20)
        if case.algorithmic_bytes > 129e6 else
        "working set fits in L2: a 256 MB write flushes L2 before every launch, outside the timed spans",
        "parallelism": "replicas x%d (each GPU its own full GEMM)" % n_gpus,
    }


# ----------------------------------------------------------------------------
# host-side arithmetic of the measurements (no GPU; tested on the CPU)


def tile_covering_entries(M, N, row_block=128, col_block=256):
    """The tile-covering sample of an M x N output: one full row in every
    row_block-row block and one full column in every col_block-column block
    (the row's position within its block varies from block to block, as
    does the column's), each output element listed once.  Every
    row_block x col_block output tile holds sampled elements.  Returns
    (rows, cols) int64 arrays."""
    import numpy as np
    pick_r = np.array(sorted({min(M - 1, b * row_block + (b * 53 + 17) % row_block)
                              for b in range((M + row_block - 1) // row_block)}), dtype=np.int64)
    pick_c = np.array(sorted({min(N - 1, b * col_block + (b * 97 + 31) % col_block)
                              for b in range((N + col_block - 1) // col_block)}), dtype=np.int64)
    r1 = np.repeat(pick_r, N)
    c1 = np.tile(np.arange(N, dtype=np.int64), len(pick_r))
    others = np.setdiff1d(np.arange(M, dtype=np.int64), pick_r)
    r2 = np.tile(others, len(pick_c))
    c2 = np.repeat(pick_c, len(others))
    return np.concatenate([r1, r2]), np.concatenate([c1, c2])


def every_nth(n_total, n_keep):
    """Indices of n_keep entries spread evenly over n_total (all when
    n_keep >= n_total)."""
    import numpy as np
    if n_keep >= n_total:
        return np.arange(n_total, dtype=np.int64)
    return np.unique(np.linspace(0, n_total - 1, max(1, n_keep)).round().astype(np.int64))


def clock_bins(chunks, width_mhz=50.0):
    """Chunks of launches grouped by the SM clock they ran at.  ``chunks``
    are dicts with ``mhz`` (probed clock), ``launches`` and ``ms`` (device
    time of the chunk).  Returns one dict per occupied bin: its clock range,
    chunk and launch counts, and the mean time per launch in the bin."""
    bins = {}
    for c in chunks:
        b = int(c["mhz"] // width_mhz)
        e = bins.setdefault(b, {"chunks": 0, "launches": 0, "ms": 0.0, "mhz_sum": 0.0})
        e["chunks"] += 1
        e["launches"] += c["launches"]
        e["ms"] += c["ms"]
        e["mhz_sum"] += c["mhz"] * c["launches"]
    out = []
    for b in sorted(bins):
        e = bins[b]
        out.append({"mhz_lo": b * width_mhz, "mhz_hi": (b + 1) * width_mhz, "chunks": e["chunks"],
                    "launches": e["launches"], "ms_per_launch": e["ms"] / e["launches"],
                    "mhz_mean": e["mhz_sum"] / e["launches"]})
    return out


def roofline_of(flops, nbytes, seconds, tensor_peak_tflops, hbm_gbs):
    """The bound of one launch of `flops` flops moving `nbytes` algorithmic
    bytes, and the fraction of that bound reached in `seconds`: "tensor"
    when the arithmetic intensity is at or above the ridge point (peak flop/s
    over copy bandwidth), else "hbm"; "latency" is added as the limit when
    the roofline time is under 3 us (launch latency dominates)."""
    t_tensor = flops / (tensor_peak_tflops * 1e12)
    t_hbm = nbytes / (hbm_gbs * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    ideal = max(t_tensor, t_hbm)
    out = {"bound": bound, "frac": ideal / seconds if seconds > 0 else None, "ideal_us": ideal * 1e6}
    if ideal < 3e-6:
        out["limited_by"] = "latency"
    return out


# ----------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)


_CODE = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3, "e5m2": 4, "e2m1": 5}


def _oracle_sampler(case):
    """Returns (run(n_entries) -> seconds, threads): the oracle, as it stands,
    on n_entries output elements of the workload spread over all threads."""
    import numpy as np

    import oracle.oracle as oracle
    from dense_tensor_core_02_gb300.inputs import make_inputs, make_scales

    A, B, C = make_inputs(case)
    sf = dict(zip(("sfa", "sfb"), (x.numpy() for x in make_scales(case)))) if case.mx else {}
    threads = len(os.sched_getaffinity(0))
    rng = np.random.default_rng(case.seed)

    def run(n):
        rows = rng.integers(0, case.M, size=n)
        cols = rng.integers(0, case.N, size=n)
        t0 = time.perf_counter()
        oracle.gemm_entries(A, B, C, case.M, case.N, case.K, rows, cols, transA=case.transA,
                            transB=case.transB, alpha=case.alpha, beta=case.beta,
                            in_dtype=_CODE[case.in_dtype], c_dtype=_CODE[case.out_dtype], threads=threads, **sf)
        return time.perf_counter() - t0

    return run, threads


def _calibrate(run, threads, target_s):
    n = threads * 2
    while True:
        t = run(n)
        if t >= 0.25 or n >= 1 << 24:
            return max(threads, int(n * target_s / max(t, 1e-9))), t
        n *= 4


# Workloads whose full problem the CPU table times (BASELINE order, 1-based):
# the single atom, 512^3, 4096^3 and 1000^3; the others are timed on the
# tile-covering sample.
CPU_FULL_PROBLEM = (1, 2, 3, 10)


def cpu_oracle_timings(case, index, A, B, C, threads, budget_s):
    """The oracle as it stands on this workload, on one thread and on
    `threads` threads: the full problem (CPU_FULL_PROBLEM) or the
    tile-covering sample.  A run whose projected time exceeds its share of
    `budget_s` is cut to an evenly spread subset (rows of the full problem,
    entries of the sample); the full problem's time is then extrapolated
    from the measured rate and labelled "extrapolated"."""
    import numpy as np

    import oracle.oracle as oracle
    kw = dict(transA=case.transA, transB=case.transB, alpha=case.alpha, beta=case.beta,
              in_dtype=_CODE[case.in_dtype], c_dtype=_CODE[case.out_dtype])
    full = index in CPU_FULL_PROBLEM
    flop_per_entry = 2.0 * case.K
    full_flops = float(case.flops)
    # single-threaded calibration on a few entries: the per-thread rate
    rng = np.random.default_rng(case.seed)
    n_cal = int(max(16, min(case.M * case.N, 2e7 / max(flop_per_entry, 1.0))))
    cr, cc = rng.integers(0, case.M, n_cal), rng.integers(0, case.N, n_cal)
    t0 = time.perf_counter()
    oracle.gemm_entries(A, B, C, case.M, case.N, case.K, cr, cc, threads=1, **kw)
    rate1 = n_cal * flop_per_entry / max(time.perf_counter() - t0, 1e-9)
    # shares of the budget per run: the full 4096^3 problem on all cores
    # 40 %, the other all-core runs 6 % each; one thread: 8 % for a full
    # problem, 2 % for a sample
    caps = {"all": budget_s * (0.40 if index == 3 else 0.06), "single": budget_s * (0.08 if full else 0.02)}
    if not full:
        rows_s, cols_s = tile_covering_entries(case.M, case.N)
        sample_desc = ("tile-covering sample: one full row per 128-row block and one full column per "
                       "256-column block (%d output elements)" % len(rows_s))
    out = {"workload": case.name, "index": index, "threads_all": threads,
           "work": "full problem" if full else sample_desc}
    for label, nthr in (("single_thread", 1), ("all_cores", threads)):
        rate_guess = rate1 * (nthr if nthr == 1 else 0.8 * nthr)
        if full:
            rows_needed = case.M
            flops_row = 2.0 * case.N * case.K
            keep = int(min(rows_needed, max(1, caps["all" if nthr > 1 else "single"] * rate_guess / flops_row)))
            t0 = time.perf_counter()
            oracle.gemm(A, B, C, case.M, case.N, case.K, rows=(0, keep), threads=nthr, **kw)
            sec = time.perf_counter() - t0
            done = keep * flops_row
            what = "the full problem" if keep == rows_needed else "rows 0..%d of %d of the full problem" % (
                keep, rows_needed)
        else:
            n_all = len(rows_s)
            keep = int(min(n_all, max(nthr * 4, caps["all" if nthr > 1 else "single"] * rate_guess /
                                      flop_per_entry)))
            idx = every_nth(n_all, keep)
            t0 = time.perf_counter()
            oracle.gemm_entries(A, B, C, case.M, case.N, case.K, rows_s[idx], cols_s[idx], threads=nthr, **kw)
            sec = time.perf_counter() - t0
            done = len(idx) * flop_per_entry
            what = "the whole sample" if len(idx) == n_all else "%d of its elements, evenly spread" % len(idx)
        rate = done / sec
        out[label] = {"threads": nthr, "measured_on": what, "seconds": sec, "gflops": rate / 1e9,
                      "full_problem_seconds": full_flops / rate,
                      "full_problem_seconds_kind": "measured" if (full and done == full_flops) else "extrapolated"}
    return out


def run_reference(args, case):
    rank, world, _ = _rank_info()
    if rank != 0:
        return 0
    run, threads = _oracle_sampler(case)
    per_step_s = min(0.25, 90.0 / max(1, args.steps + args.warmup))
    n, _ = _calibrate(run, threads, per_step_s)
    for _ in range(args.warmup):
        run(n)
    total = 0.0
    for _ in range(args.steps):
        total += run(n)
    flops = 2.0 * case.K * n * args.steps
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _workload_config(case, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "each step: %d output elements of %s (full K=%d dot products)" % (
                             n, case.name, case.K)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# the CUDA path

CLOCK_CHUNK = 16                # launches per chunk of the clock study
GRAPH_LAUNCHES = 50             # launches per CUDA graph of a per-config row that fits in L2
FLUSH_BYTES = 256 << 20         # the L2 flush write (L2 is 129 MB)
SPARE_SMS = 2                   # SMs a clock measurement leaves free for its probe
PROBE_INTERVAL_NS = 20000       # one clock sample every 20 us

# Measurement helper compiled by this script (not part of the library): a
# one-thread kernel that samples (%globaltimer, %clock64, %smid) every
# interval_ns, n times (so it ends after n * interval_ns), and a one-thread
# kernel that writes %globaltimer once, to mark where a loop starts and ends
# on the same clock.  An SM's clock64 advances at that SM's clock, so the
# ratio of the two counters between samples is the clock the SMs ran at.
_CLOCK_PROBE_SRC = r"""
#include <cuda_runtime.h>
__global__ void gb_clock_probe(unsigned long long* out, int n, unsigned long long interval_ns) {
    unsigned long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (int i = 0; i < n; ++i) {
        unsigned long long t;
        do {
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        } while (t < t0 + (unsigned long long)i * interval_ns);
        unsigned long long c = clock64();
        unsigned int sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        out[3 * i] = t;
        out[3 * i + 1] = c;
        out[3 * i + 2] = sm;
    }
}
__global__ void gb_stamp(unsigned long long* out) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    *out = t;
}
extern "C" int launch_clock_probe(void* out, int n, unsigned long long interval_ns, void* stream) {
    gb_clock_probe<<<1, 1, 0, (cudaStream_t)stream>>>((unsigned long long*)out, n, interval_ns);
    return (int)cudaGetLastError();
}
extern "C" int launch_stamp(void* out, void* stream) {
    gb_stamp<<<1, 1, 0, (cudaStream_t)stream>>>((unsigned long long*)out);
    return (int)cudaGetLastError();
}
"""


def load_clock_probe():
    """Compiles the measurement helper above with nvcc into a temporary
    directory and loads it; None if that fails (the clock is then not
    reported)."""
    import ctypes
    import shutil
    import tempfile
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    d = tempfile.mkdtemp(prefix="gemm_bench_probe_")
    src, lib = os.path.join(d, "probe.cu"), os.path.join(d, "libprobe.so")
    with open(src, "w") as f:
        f.write(_CLOCK_PROBE_SRC)
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                        "-o", lib, src], capture_output=True, text=True)
    if r.returncode != 0:
        shutil.rmtree(d, ignore_errors=True)
        return None
    probe = ctypes.CDLL(lib)
    shutil.rmtree(d, ignore_errors=True)   # the loaded library stays mapped
    probe.launch_clock_probe.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong, ctypes.c_void_p]
    probe.launch_stamp.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    # Launch both kernels once now: the first launch of a kernel loads it,
    # and that load would wait for a probe already running on the GPU.
    import torch
    scratch = torch.zeros(8, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if probe.launch_clock_probe(scratch.data_ptr(), 1, 1000, s) != 0 or probe.launch_stamp(scratch.data_ptr(), s) != 0:
        return None
    torch.cuda.synchronize()
    return probe


def clock_series(samples):
    """(time ns, MHz) between consecutive probe samples taken on one SM."""
    out = []
    for (t0, c0, s0), (t1, c1, s1) in zip(samples, samples[1:]):
        if t1 > t0 and s0 == s1 and c1 >= c0:
            out.append((0.5 * (t0 + t1), (c1 - c0) / (t1 - t0) * 1e3))
    return out


def clock_between(series, t0, t1):
    """The clock readings whose interval centre lies in [t0, t1] (ns)."""
    return [m for t, m in series if t0 <= t <= t1]


class ClockProbe:
    """Runs loops of a workload with the persistent grid planned for
    SPARE_SMS fewer SMs while the probe kernel samples the clock on a free SM
    (a probe between launches cannot see the clock a loop runs at: the
    power limiter lets it back up within ~0.1 ms of the load stopping).
    Each loop is bracketed by timestamp kernels on its stream."""

    def __init__(self, torch, dev, num_sms, lib):
        self.torch, self.dev, self.num_sms, self.lib = torch, dev, num_sms, lib

    def run(self, wl, segments, launches_per_segment, fits_l2=False, flush=None):
        """`segments` back-to-back segments of `launches_per_segment` launches
        after an idle pause of 0.5 s.  Returns (per-segment list of (device
        ms per launch, median MHz, readings)) or None."""
        torch = self.torch
        old = os.environ.get("GEMM_MAX_SMS")
        os.environ["GEMM_MAX_SMS"] = str(self.num_sms - SPARE_SMS)
        try:
            s1, s2 = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
            sptr = s1.cuda_stream
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s1):
                for _ in range(3):
                    wl.step(sptr)
                e0.record(s1)
                wl.step(sptr)
                e1.record(s1)
            torch.cuda.synchronize(self.dev)
            est_ms = max(e0.elapsed_time(e1), 1e-3) * (2.0 if fits_l2 else 1.0)
            total_ms = est_ms * segments * launches_per_segment * 1.5 + 20.0
            n = int(total_ms * 1e6 / PROBE_INTERVAL_NS) + 10
            buf = torch.zeros(3 * n, dtype=torch.int64, device=self.dev)
            stamps = torch.zeros(segments + 1, dtype=torch.int64, device=self.dev)
            spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(segments)]
            time.sleep(0.5)
            if self.lib.launch_clock_probe(buf.data_ptr(), n, PROBE_INTERVAL_NS, s2.cuda_stream) != 0:
                return None
            time.sleep(0.002)   # the probe is running before the loop starts
            with torch.cuda.stream(s1):
                for k, (a, b) in enumerate(spans):
                    if self.lib.launch_stamp(stamps[k:].data_ptr(), sptr) != 0:
                        return None
                    a.record(s1)
                    for _ in range(launches_per_segment):
                        if fits_l2:
                            flush.zero_()
                        wl.step(sptr)
                    b.record(s1)
                if self.lib.launch_stamp(stamps[segments:].data_ptr(), sptr) != 0:
                    return None
            torch.cuda.synchronize(self.dev)
            series = clock_series([tuple(x) for x in buf.view(-1, 3).cpu().tolist()])
            st = stamps.cpu().tolist()
            out = []
            for k, (a, b) in enumerate(spans):
                inside = clock_between(series, st[k], st[k + 1])
                out.append((a.elapsed_time(b) / launches_per_segment,
                            statistics.median(inside) if inside else None, len(inside)))
            return out
        finally:
            if old is None:
                os.environ.pop("GEMM_MAX_SMS", None)
            else:
                os.environ["GEMM_MAX_SMS"] = old


def clock_during(probe, wl, launches, fits_l2=False, flush=None):
    """The SM clock during a loop of `launches` launches (the loop run again
    beside the clock probe after an idle pause): (median MHz, readings)."""
    if probe is None:
        return None, 0
    res = probe.run(wl, 1, launches, fits_l2, flush)
    if not res or res[0][1] is None:
        return None, 0
    return res[0][1], res[0][2]


class _Workload:
    """One workload's device buffers and its launch through the C ABI."""

    def __init__(self, case, dev, host=None):
        import torch

        from dense_tensor_core_02_gb300 import binding
        from dense_tensor_core_02_gb300.inputs import make_inputs, make_scales
        self.case, self.binding = case, binding
        self.code = {"f16": binding.F16, "bf16": binding.BF16, "f32": binding.F32, "e4m3": binding.E4M3,
                     "e5m2": binding.E5M2, "e2m1": binding.E2M1}
        self.epu = 2 if case.in_dtype == "e2m1" else 1   # operand elements per stored byte (packed fp4)
        self.A, self.B, self.C = host if host is not None else make_inputs(case)
        self.SFA, self.SFB = make_scales(case) if case.mx else (None, None)
        self.Ad, self.Bd = self.A.to(dev), self.B.to(dev)
        self.Cd = self.C.to(dev) if self.C is not None else None
        self.SFAd = self.SFA.to(dev) if self.SFA is not None else None
        self.SFBd = self.SFB.to(dev) if self.SFB is not None else None
        self.otype = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[case.out_dtype]
        self.Dd = torch.empty((case.M, case.N), dtype=self.otype, device=dev)
        # launches per step: gemm_mx rearranges both operands' scales first (one launch)
        self.launches_per_step = 2 if case.mx else 1

    def call(self, D_, A_, B_, C_, SFA_, SFB_, s_ptr):
        case, b = self.case, self.binding
        if case.mx:
            rc = b.gemm_mx(D_, A_, B_, C_, SFA_, SFB_, case.M, case.N, case.K, A_.stride(0) * self.epu,
                           B_.stride(0) * self.epu, C_.stride(0) if C_ is not None else case.N, D_.stride(0),
                           SFA_.stride(0), SFB_.stride(0), case.transA, case.transB, case.alpha, case.beta,
                           self.code[case.in_dtype], self.code[case.out_dtype], s_ptr)
        else:
            rc = b.gemm(D_, A_, B_, C_, case.M, case.N, case.K, A_.stride(0), B_.stride(0),
                        C_.stride(0) if C_ is not None else case.N, D_.stride(0), case.transA, case.transB,
                        case.alpha, case.beta, self.code[case.in_dtype], self.code[case.out_dtype], s_ptr)
        if rc != 0:
            raise RuntimeError("gemm: %s" % b.gemm_status_string(rc))

    def step(self, s_ptr):
        self.call(self.Dd, self.Ad, self.Bd, self.Cd, self.SFAd, self.SFBd, s_ptr)


def _event_pair(torch):
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def clock_study(torch, probe, wl, dev, seconds, num_sms, rate):
    """The workload back to back for about `seconds` after an idle pause, in
    chunks of CLOCK_CHUNK launches between CUDA events, beside the clock
    probe (ClockProbe): per chunk the device time per launch and the median
    clock inside it.  Returns the chunk table's summary and its bins by
    clock, or None without the probe."""
    if probe is None:
        return None
    sptr = torch.cuda.current_stream(dev).cuda_stream
    e0, e1 = _event_pair(torch)
    e0.record()
    for _ in range(CLOCK_CHUNK):
        wl.step(sptr)
    e1.record()
    torch.cuda.synchronize(dev)
    chunk_ms = max(e0.elapsed_time(e1), 1e-3)
    n_chunks = max(8, min(2000, int(seconds * 1e3 / chunk_ms)))
    res = probe.run(wl, n_chunks, CLOCK_CHUNK)
    if not res:
        return None
    chunks = [{"mhz": m, "launches": CLOCK_CHUNK, "ms": ms * CLOCK_CHUNK, "readings": r}
              for ms, m, r in res if m]
    if not chunks:
        return None
    sms = num_sms - SPARE_SMS
    flops = wl.case.flops
    ideal_cycles = flops / (sms * FLOP_PER_CLK_PER_SM * rate)
    total_ms = sum(c["ms"] for c in chunks)
    launches = sum(c["launches"] for c in chunks)
    mhz = [c["mhz"] for c in chunks]
    cyc = [c["ms"] / c["launches"] * 1e-3 * c["mhz"] * 1e6 for c in chunks]
    med_mhz = statistics.median(mhz)
    ms_per_launch = total_ms / launches
    achieved = flops / (ms_per_launch * 1e-3) / 1e12
    clk_peak = sms * FLOP_PER_CLK_PER_SM * rate * med_mhz * 1e6 / 1e12
    bins = clock_bins(chunks)
    for bn in bins:
        t = bn["ms_per_launch"] * 1e-3
        bn["tflops"] = flops / t / 1e12
        bn["cycles_per_launch"] = t * bn["mhz_mean"] * 1e6
        bn["frac_of_clock_peak"] = ideal_cycles / bn["cycles_per_launch"]
    first = chunks[0]
    return {
        "launches": launches, "chunks": len(chunks), "seconds": total_ms * 1e-3, "sms": sms,
        "clock_readings": sum(c["readings"] for c in chunks),
        "method": "a one-thread probe kernel samples %%globaltimer and %%clock64 every %d us on one of the %d SMs "
                  "the grid leaves free; timestamp kernels between chunks place them on the same clock; a "
                  "chunk's clock is the median reading inside it" % (PROBE_INTERVAL_NS // 1000, SPARE_SMS),
        "ms_per_launch": ms_per_launch, "tflops": achieved,
        "sm_mhz_median": med_mhz, "sm_mhz_min": min(mhz), "sm_mhz_max": max(mhz),
        "clock_peak_tflops_at_median": clk_peak, "frac_of_clock_peak": achieved / clk_peak,
        "cycles_per_launch_median": statistics.median(cyc), "ideal_cycles_per_launch": ideal_cycles,
        "first_chunk": {"sm_mhz": first["mhz"], "ms_per_launch": first["ms"] / first["launches"],
                        "frac_of_clock_peak": ideal_cycles / (first["ms"] / first["launches"] * 1e-3 *
                                                              first["mhz"] * 1e6)},
        "bins": bins,
    }


def per_config_row(torch, case, index, dev, stream, peaks, num_sms, flush, probe=None):
    """One BASELINE workload: 10 warm-ups, then >= 50 launches and >= 200 ms.
    Workloads larger than L2 run back to back in 5 groups between events
    (median and min over the groups' time per launch); workloads that fit
    in L2 get an L2 flush before every launch, each launch between its own
    events (median and min over launches).  The clock the loop ran at is
    measured while it runs again beside the clock probe (clock_during)."""
    wl = _Workload(case, dev)
    sptr = stream.cuda_stream
    fits_l2 = case.algorithmic_bytes <= 129e6
    w0, w1 = _event_pair(torch)
    with torch.cuda.stream(stream):
        w0.record(stream)
        for _ in range(10):
            wl.step(sptr)
        w1.record(stream)
    torch.cuda.synchronize(dev)
    est_ms = max(w0.elapsed_time(w1) / 10, 1e-3)
    n = int(min(5000, max(50, 200.0 / est_ms)))
    with torch.cuda.stream(stream):
        if fits_l2:
            spans = [_event_pair(torch) for _ in range(n)]
            for a, b in spans:
                flush.zero_()
                a.record(stream)
                wl.step(sptr)
                b.record(stream)
        else:
            groups = 5
            per = (n + groups - 1) // groups
            spans = [_event_pair(torch) for _ in range(groups)]
            for a, b in spans:
                a.record(stream)
                for _ in range(per):
                    wl.step(sptr)
                b.record(stream)
    torch.cuda.synchronize(dev)
    # Workloads that fit in L2 are a launch and a few memory latencies: their
    # time per launch back to back, warm, with the host out of the way
    # (GRAPH_LAUNCHES calls captured into one CUDA graph, best of 3 replays).
    graph_us = None
    if fits_l2:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for _ in range(GRAPH_LAUNCHES):
                wl.step(sptr)
        with torch.cuda.stream(stream):
            g.replay()
            reps = [_event_pair(torch) for _ in range(3)]
            for a, b in reps:
                a.record(stream)
                g.replay()
                b.record(stream)
        torch.cuda.synchronize(dev)
        graph_us = min(a.elapsed_time(b) for a, b in reps) * 1e3 / GRAPH_LAUNCHES
        del g
    status, info = wl.binding.gemm_poll_device_error(stream)
    if status != 0:
        raise RuntimeError("device status after %s: %s %s" % (case.name, wl.binding.gemm_status_string(status),
                                                               info))
    if fits_l2:
        per_launch = [a.elapsed_time(b) for a, b in spans]
        launches = n
    else:
        per_launch = [a.elapsed_time(b) / per for a, b in spans]
        launches = per * len(spans)
    med, mn = statistics.median(per_launch), min(per_launch)
    rate = FP8_RATE if case.in_dtype in ("e4m3", "e5m2", "e2m1") else 1.0
    peak_burst = float(peaks["bf16_tflops"]) * rate
    hbm = float(peaks["hbm_gbs"])
    roof = roofline_of(case.flops, case.algorithmic_bytes, med * 1e-3, peak_burst, hbm)
    during, n_samples = clock_during(probe, wl, launches, fits_l2, flush)
    mhz = [during] if during else []
    row = {
        "index": index, "workload": case.name,
        "M": case.M, "N": case.N, "K": case.K, "in_dtype": case.in_dtype, "out_dtype": case.out_dtype,
        "alpha": case.alpha, "beta": case.beta, "transA": case.transA, "transB": case.transB,
        "launches": launches, "timing": ("each launch between its own events after a 256 MB L2 flush"
                                         if fits_l2 else "5 groups of back-to-back launches between events"),
        "us_median": med * 1e3, "us_min": mn * 1e3, "us_graph_replayed": graph_us,
        "tflops_median": case.flops / (med * 1e-3) / 1e12, "tflops_best": case.flops / (mn * 1e-3) / 1e12,
        "gbs_median": case.algorithmic_bytes / (med * 1e-3) / 1e9,
        "algorithmic_flops": case.flops, "algorithmic_bytes": case.algorithmic_bytes,
        "bound": roof["bound"], "frac": roof["frac"], "roofline_ideal_us": roof["ideal_us"],
        "peak": peak_burst if roof["bound"] == "tensor" else hbm,
        "peak_unit": UNIT if roof["bound"] == "tensor" else "GB/s",
        "peak_kind": ("measured bf16 burst (cuBLAS)" + ("" if rate == 1.0 else " x 2, nominal fp8 / bf16 ratio"))
        if roof["bound"] == "tensor" else "measured HBM copy bandwidth",
        "sm_mhz_during": statistics.mean(mhz) if mhz else None,
        "clock_samples": n_samples,
        "traffic": _profiled_traffic(case.name),
        "ncu_us": _profiled_duration_us(case.name),
    }
    if row["ncu_us"] and roof["bound"] == "tensor":
        # the committed ncu launch (one serialised launch) against the same peak
        row["frac_ncu"] = case.flops / (row["ncu_us"] * 1e-6) / 1e12 / peak_burst
    if "limited_by" in roof:
        row["limited_by"] = roof["limited_by"]
    if mhz and roof["bound"] == "tensor":
        row["frac_of_clock_peak"] = row["tflops_median"] / (
            num_sms * FLOP_PER_CLK_PER_SM * rate * statistics.mean(mhz) * 1e6 / 1e12)
    host = (wl.A, wl.B, wl.C)
    del wl
    return row, host


def run_ours(args, case):
    import torch

    from dense_tensor_core_02_gb300 import binding
    from dense_tensor_core_02_gb300.inputs import CASES

    rank, world, local_rank = _rank_info()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    binding.load_library()

    wl = _Workload(case, dev)
    A, B, C, SFA, SFB = wl.A, wl.B, wl.C, wl.SFA, wl.SFB
    Dd, otype = wl.Dd, wl.otype
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    small = case.algorithmic_bytes <= 129e6
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        wl.step(sptr)

    def barrier():
        if dist is not None:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    status, info = binding.gemm_poll_device_error(stream)
    if status != 0:
        raise RuntimeError("device status after warm-up: %s %s" % (binding.gemm_status_string(status), info))

    def timed(n):
        """Device time (ms) of n launches on the stream.  Working sets that
        fit in L2 get a flush (a 256 MB write) before every launch, outside
        the timed spans: each launch is bracketed by its own event pair."""
        with torch.cuda.stream(stream):
            if not small:
                e0.record(stream)
                for _ in range(n):
                    step()
                e1.record(stream)
            else:
                spans = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                         for _ in range(n)]
                for a, b in spans:
                    flush.zero_()
                    a.record(stream)
                    step()
                    b.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) if not small else sum(a.elapsed_time(b) for a, b in spans)

    # burst: the best of three runs of BURST_STEPS launches, measured the way
    # the burst peak is (a short run after an idle pause, before the power cap
    # sets in); the headline is the run below
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    burst_runs = []
    for _ in range(3):
        time.sleep(0.2)   # let the power state settle back between runs
        burst_runs.append(timed(BURST_STEPS) / BURST_STEPS)
    burst_ms = min(burst_runs)

    sampler = ClockSampler(local_rank).start() if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    barrier()
    torch.cuda.synchronize(dev)
    elapsed_ms = timed(args.steps)
    barrier()
    # after the timed region, on rank 0 at N = 1, with the sampler still
    # running (its samples then cover all of it): the clock the timed loop
    # ran at (the same loop again, its clock read by NVML while it runs),
    # the same for a burst, then the clock study
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rate = FP8_RATE if case.in_dtype in ("e4m3", "e5m2", "e2m1") else 1.0
    study = None
    timed_mhz, timed_samples, burst_mhz = None, 0, None
    probe = None
    if world == 1 and not args.no_clock_study:
        lib = load_clock_probe()
        probe = ClockProbe(torch, dev, num_sms, lib) if lib is not None else None
        timed_mhz, timed_samples = clock_during(probe, wl, args.steps, small, flush)
        burst_mhz, _ = clock_during(probe, wl, BURST_STEPS, small, flush)
        if not small:
            study = clock_study(torch, probe, wl, dev, args.clock_study_seconds, num_sms, rate)
    clocks = sampler.stop() if sampler else None
    if clocks is not None:
        clocks["sm_mhz_during_timed_loop"] = timed_mhz
        clocks["sm_mhz_during_timed_loop_samples"] = timed_samples
        clocks["window"] = ("the timed region (%.0f ms)%s" % (
            elapsed_ms, " and the clock measurements after it (%.1f s)" % (study["seconds"] if study else 0.0)))
    status, info = binding.gemm_poll_device_error(stream)
    if status != 0:
        raise RuntimeError("device status after timing: %s %s" % (binding.gemm_status_string(status), info))
    elapsed_ms = slowest_rank_ms(elapsed_ms, dist, dev)

    per_launch_ms = elapsed_ms / args.steps
    value = job_tflops(world, case.flops, args.steps, elapsed_ms)

    # end to end through the C ABI's host-buffer entry point gemm_host():
    # pinned host inputs in, host result out, every copy inside the timed
    # region (each call stages and pipelines them over row panels of D).
    # Consecutive steps alternate between E2E_STREAMS streams, each with its
    # own result buffer and staging, so that one step's copy-in overlaps the
    # previous step's copy-out as in a job that streams independent problems;
    # the timed region runs from before the first step on every stream to
    # after the last step on every stream.
    e2e = None
    if not args.no_e2e:
        hA = A.pin_memory()
        hB = B.pin_memory()
        hC = C.pin_memory() if C is not None else None
        streams = [torch.cuda.Stream(dev) for _ in range(E2E_STREAMS)]
        hDs = [torch.empty((case.M, case.N), dtype=otype).pin_memory() for _ in streams]
        if case.mx:
            # gemm_mx takes device buffers: each step copies its inputs in and
            # its result out on its stream around the call (no panelling)
            hSFA, hSFB = SFA.pin_memory(), SFB.pin_memory()
            dbufs = [[torch.empty_like(x, device=dev) if x is not None else None
                      for x in (hD, hA, hB, hC, hSFA, hSFB)] for hD in hDs]

        def e2e_step(i):
            s_i, hD = streams[i % len(streams)], hDs[i % len(streams)]
            if case.mx:
                dD, dA, dB, dC, dSA, dSB = dbufs[i % len(streams)]
                with torch.cuda.stream(s_i):
                    for d_, h_ in ((dA, hA), (dB, hB), (dC, hC), (dSA, hSFA), (dSB, hSFB)):
                        if d_ is not None:
                            d_.copy_(h_, non_blocking=True)
                    wl.call(dD, dA, dB, dC, dSA, dSB, s_i.cuda_stream)
                    hD.copy_(dD, non_blocking=True)
                return
            rc = binding.gemm_host(hD, hA, hB, hC, case.M, case.N, case.K, hA.stride(0), hB.stride(0),
                                   hC.stride(0) if hC is not None else case.N, hD.stride(0), case.transA,
                                   case.transB, case.alpha, case.beta, wl.code[case.in_dtype],
                                   wl.code[case.out_dtype], s_i.cuda_stream)
            if rc != 0:
                raise RuntimeError("gemm_host: %s" % binding.gemm_status_string(rc))

        for i in range(2 * len(streams)):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in streams]
        ends = [torch.cuda.Event(enable_timing=True) for _ in streams]
        for st, ev in zip(streams, starts):
            ev.record(st)
        for i in range(args.e2e_steps):
            e2e_step(i)
        for st, ev in zip(streams, ends):
            ev.record(st)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = max(starts[0].elapsed_time(e) for e in ends) - min(starts[0].elapsed_time(e) for e in starts)
        e2e_ms = slowest_rank_ms(e2e_ms, dist, dev)
        ref = hDs[0]
        for hD in hDs[1:]:   # every stream computed the same product
            if not torch.equal(hD, ref):
                raise RuntimeError("end-to-end results differ between streams")
        h2d = A.numel() * A.element_size() + B.numel() * B.element_size() + (
            C.numel() * C.element_size() if C is not None else 0) + (
            SFA.numel() + SFB.numel() if case.mx else 0)
        d2h = Dd.numel() * Dd.element_size()
        e2e = {"value": job_tflops(world, case.flops, args.e2e_steps, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "ms_per_step": e2e_ms / args.e2e_steps,
               "api": ("gemm_mx between a copy of the inputs in and of D out (pinned host buffers), steps "
                       "alternating between %d streams" if case.mx else
                       "gemm_host (pinned host buffers; copies pipelined with the products over row panels; "
                       "steps alternate between %d streams)") % len(streams)}
        del hA, hB, hC, hDs, streams

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = _measured_peaks()
    achieved = case.flops / (per_launch_ms * 1e-3) / 1e12
    # 8-bit operands: no measured fp8 peak exists, so the measured bf16 figures
    # are scaled by the nominal dense fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s).
    # Packed 4-bit operands run on the same kind::mxf8f6f4 instruction as the
    # 8-bit ones (K = 32 per instruction), so their peak is the 8-bit one.
    peak_burst = float(peaks["bf16_tflops"]) * rate
    peak_sustained = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * rate
    # The measured peaks come as a burst (a short cuBLAS run, clocks up) and a
    # sustained figure (seconds of back-to-back cuBLAS under the power cap).
    # The timed loop is held to the same condition as its denominator: a loop
    # that ran long enough to meet the power cap (>= 0.5 s) is compared with
    # the sustained peak; a short loop, and the burst figure, with the burst
    # peak.
    power_capped = elapsed_ms >= 500.0
    peak = peak_sustained if power_capped else peak_burst
    kind = "sustained" if power_capped else "burst"
    src = ("%s bf16 %s (cuBLAS 8192^3, MEASURED_PEAKS.json)%s; this loop: %d launches in %.0f ms" % (
        peak_src, kind, "; f16 runs at the bf16 rate" if rate == 1.0 else
        " x 2, the nominal dense fp8 / bf16 ratio", args.steps, elapsed_ms))
    achieved_gbs = case.algorithmic_bytes / (per_launch_ms * 1e-3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    # the bound: below the ridge (peak flop/s / copy bandwidth) the algorithmic
    # bytes limit the launch, above it the tensor cores do
    intensity = case.flops / case.algorithmic_bytes
    ridge = peak_burst * 1e12 / (hbm * 1e9)
    burst_tflops = case.flops / (burst_ms * 1e-3) / 1e12
    if intensity >= ridge:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                    "frac": achieved / peak, "peak_kind": kind, "peak_source": src,
                    "frac_of_burst": achieved / peak_burst, "frac_of_sustained": achieved / peak_sustained,
                    "frac_of_nominal": achieved / (NOMINAL_DENSE_TFLOPS * rate)}
        burst = {"achieved": burst_tflops, "frac": burst_tflops / peak_burst, "peak": peak_burst}
    else:
        roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                    "frac": achieved_gbs / hbm,
                    "peak_source": "%s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_src,
                    "achieved_tflops": achieved, "tensor_peak_tflops": peak_burst}
        burst_gbs = case.algorithmic_bytes / (burst_ms * 1e-3) / 1e9
        burst = {"achieved": burst_gbs, "frac": burst_gbs / hbm}
    roofline.update({"traffic": _profiled_traffic(case.name), "arithmetic_intensity": intensity,
                     "ridge_flop_per_byte": ridge, "algorithmic_flops_per_launch": case.flops,
                     "algorithmic_bytes_per_launch": case.algorithmic_bytes, "achieved_gbs": achieved_gbs})
    roofline["burst"] = dict(burst, launches=BURST_STEPS, best_of=3, ms_per_launch=burst_ms, sm_mhz_during=burst_mhz)
    if case.mx:
        roofline["note"] = ("block-scaled: the time per launch is that of the whole gemm_mx step, the two small "
                            "scale-rearranging launches included" +
                            ("; packed E2M1 runs on kind::mxf8f6f4 at the 8-bit instruction rate, so the peak is "
                             "the 8-bit one" if case.in_dtype == "e2m1" else ""))
    if roofline["bound"] == "tensor":
        # the dense peak at the clock the launches ran at: n_SM x 8192 flop/clk x f
        # (x 2 for 8-bit operands), with f from the clock probes -- the one before
        # the burst runs for the burst figure, the clock study's median for the loop
        if burst_mhz:
            roofline["burst"]["frac_of_clock_peak"] = burst_tflops / (
                num_sms * FLOP_PER_CLK_PER_SM * rate * burst_mhz * 1e6 / 1e12)
        if timed_mhz:
            # the timed loop against the dense peak at the clock it ran at
            clk_peak = num_sms * FLOP_PER_CLK_PER_SM * rate * timed_mhz * 1e6 / 1e12
            roofline["frac_of_clock_peak"] = achieved / clk_peak
            roofline["clock_peak_tflops"] = clk_peak
            roofline["clock_source"] = (
                "median of %d in-kernel clock readings on a spare SM during a repeat of the timed loop planned "
                "for %d SMs (%.0f MHz)" % (timed_samples, num_sms - SPARE_SMS, timed_mhz))
        if study:
            roofline["frac_of_clock_peak_clock_study"] = study["frac_of_clock_peak"]
    roofline["max_clock_peak_tflops"] = num_sms * FLOP_PER_CLK_PER_SM * rate * 2070e6 / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_launch_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": case.in_dtype, "data": "synthetic",
        "config": _workload_config(case, world), "roofline": roofline,
        "clocks": clocks, "e2e": e2e, "gpu_launches": args.steps * wl.launches_per_step, "num_sms": num_sms,
    }
    if study:
        line["clock_study"] = study
    del wl

    # every BASELINE workload, and the CPU oracle on the same inputs
    per_config, cpu_rows = [], []
    want_cpu = not args.no_cpu_baseline and world == 1
    if world == 1 and not args.no_per_config:
        for i, c in enumerate(CASES[:10]):
            row, host = per_config_row(torch, c, i + 1, dev, stream, peaks, num_sms, flush, probe)
            per_config.append(row)
            if want_cpu:
                cpu_rows.append(cpu_oracle_timings(c, i + 1, *host, threads=len(os.sched_getaffinity(0)),
                                                   budget_s=args.cpu_budget))
            del host
        line["per_config"] = per_config
    if want_cpu:
        head = next((r for r in cpu_rows if r["workload"] == case.name), None)
        if head is None:
            from dense_tensor_core_02_gb300.inputs import make_inputs
            head = cpu_oracle_timings(case, CASES.index(case) + 1, *make_inputs(case),
                                      threads=len(os.sched_getaffinity(0)), budget_s=args.cpu_budget)
        allc, one = head["all_cores"], head["single_thread"]
        line["cpu_baseline"] = {
            "value": allc["gflops"] / 1e3, "unit": UNIT, "cores": allc["threads"], "kind": "oracle",
            "sample": "%s of %s: %s, on %d threads (%.1f s)" % (head["work"], case.name, allc["measured_on"],
                                                                 allc["threads"], allc["seconds"]),
            "single_thread_value": one["gflops"] / 1e3,
            "single_thread_sample": "%s, on 1 thread (%.1f s)" % (one["measured_on"], one["seconds"]),
            "full_problem_seconds_all_cores": allc["full_problem_seconds"],
            "full_problem_seconds_all_cores_kind": allc["full_problem_seconds_kind"],
            "full_problem_seconds_single_thread": one["full_problem_seconds"],
            "full_problem_seconds_single_thread_kind": one["full_problem_seconds_kind"],
            "per_config": cpu_rows,
        }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = _args()
    from dense_tensor_core_02_gb300.inputs import CASE_BY_NAME, HEADLINE
    case = CASE_BY_NAME[args.case] if args.case else HEADLINE
    if args.library_peaks:
        return library_peaks()
    if args.impl == "reference":
        return run_reference(args, case)
    return run_ours(args, case)


if __name__ == "__main__":
    sys.exit(main())
