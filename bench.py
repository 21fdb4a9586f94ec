"""Throughput of D = alpha * op(A) @ op(B) + beta * C on GB300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--case NAME] [--no-e2e] [--no-cpu-baseline]

A step is one GEMM call through the C ABI over the resident, seeded
synthetic inputs of the workload (default: M = N = K = 8192, fp16
operands drawn N(0, 1/sqrt(K)), alpha = 1, beta = 0, fp32 D).  The timed
region is exactly K steps between CUDA events on the launching stream,
bracketed by a barrier and a device synchronisation; with N > 1 (torchrun)
every rank runs its own replica and the slowest rank's time is used.

The roofline's tensor peak is the measured cuBLAS bf16 figure (x 2 for
8-bit operands) in the power state the timed loop ran in: the sustained
figure for a loop long enough to meet the power cap (the default 1000
launches of the 8192^3 workload), the burst figure for a short loop and for
the separate burst measurement (best of three 10-launch runs).

--impl reference times the CPU oracle instead (the only other
implementation of this operation in the repository), on bounded samples
of the same workload, on the host cores.
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


def _profiled_traffic(case_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic_%s.txt" % case_name)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
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
                 "--format=csv,noheader,nounits", "-lms", "100"],
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
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target wall time of the CPU-baseline sample")
    return ap.parse_args()


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
# CPU oracle timing (the cpu_baseline leg and the reference arm)


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
    code = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3, "e5m2": 4, "e2m1": 5}

    def run(n):
        rows = rng.integers(0, case.M, size=n)
        cols = rng.integers(0, case.N, size=n)
        t0 = time.perf_counter()
        oracle.gemm_entries(A, B, C, case.M, case.N, case.K, rows, cols, transA=case.transA,
                            transB=case.transB, alpha=case.alpha, beta=case.beta,
                            in_dtype=code[case.in_dtype], c_dtype=code[case.out_dtype], threads=threads, **sf)
        return time.perf_counter() - t0

    return run, threads


def _calibrate(run, threads, target_s):
    n = threads * 2
    while True:
        t = run(n)
        if t >= 0.25 or n >= 1 << 24:
            return max(threads, int(n * target_s / max(t, 1e-9))), t
        n *= 4


def cpu_baseline(case, target_s):
    run, threads = _oracle_sampler(case)
    n, _ = _calibrate(run, threads, target_s)
    t = run(n)
    flops = 2.0 * case.K * n
    return {"value": flops / t / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d output elements of %s (random positions, each the full K=%d dot product), "
                      "%.1f s on %d threads" % (n, case.name, case.K, t, threads)}


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


def run_ours(args, case):
    import torch

    from dense_tensor_core_02_gb300 import binding
    from dense_tensor_core_02_gb300.inputs import make_inputs, make_scales

    rank, world, local_rank = _rank_info()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    binding.load_library()

    code = {"f16": binding.F16, "bf16": binding.BF16, "f32": binding.F32, "e4m3": binding.E4M3,
            "e5m2": binding.E5M2, "e2m1": binding.E2M1}
    epu = 2 if case.in_dtype == "e2m1" else 1   # operand elements per stored byte (packed fp4)
    A, B, C = make_inputs(case)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = C.to(dev) if C is not None else None
    SFA, SFB = make_scales(case) if case.mx else (None, None)
    SFAd = SFA.to(dev) if SFA is not None else None
    SFBd = SFB.to(dev) if SFB is not None else None
    # launches per step: gemm_mx rearranges both operands' scales first (one launch)
    launches_per_step = 2 if case.mx else 1
    otype = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[case.out_dtype]
    Dd = torch.empty((case.M, case.N), dtype=otype, device=dev)
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    ldc = Cd.stride(0) if Cd is not None else case.N
    small = case.algorithmic_bytes <= 129e6
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if small else None

    def call(D_, A_, B_, C_, SFA_, SFB_, s_ptr):
        if case.mx:
            rc = binding.gemm_mx(D_, A_, B_, C_, SFA_, SFB_, case.M, case.N, case.K, A_.stride(0) * epu,
                                 B_.stride(0) * epu,
                                 C_.stride(0) if C_ is not None else case.N, D_.stride(0), SFA_.stride(0),
                                 SFB_.stride(0), case.transA, case.transB, case.alpha, case.beta,
                                 code[case.in_dtype], code[case.out_dtype], s_ptr)
        else:
            rc = binding.gemm(D_, A_, B_, C_, case.M, case.N, case.K, A_.stride(0), B_.stride(0),
                              C_.stride(0) if C_ is not None else case.N, D_.stride(0), case.transA, case.transB,
                              case.alpha, case.beta, code[case.in_dtype], code[case.out_dtype], s_ptr)
        if rc != 0:
            raise RuntimeError("gemm: %s" % binding.gemm_status_string(rc))

    def step():
        call(Dd, Ad, Bd, Cd, SFAd, SFBd, sptr)

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
            if flush is None:
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
        return e0.elapsed_time(e1) if flush is None else sum(a.elapsed_time(b) for a, b in spans)

    # burst: the best of three runs of BURST_STEPS launches, measured the way
    # the burst peak is (a short run, before the power cap sets in); the
    # headline is the long run below, reported against both peaks
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    burst_ms = min(timed(BURST_STEPS) for _ in range(3)) / BURST_STEPS

    sampler = ClockSampler(local_rank).start() if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    barrier()
    torch.cuda.synchronize(dev)
    elapsed_ms = timed(args.steps)
    barrier()
    clocks = sampler.stop() if sampler else None
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
                    call(dD, dA, dB, dC, dSA, dSB, s_i.cuda_stream)
                    hD.copy_(dD, non_blocking=True)
                return
            rc = binding.gemm_host(hD, hA, hB, hC, case.M, case.N, case.K, hA.stride(0), hB.stride(0),
                                   hC.stride(0) if hC is not None else case.N, hD.stride(0), case.transA,
                                   case.transB, case.alpha, case.beta, code[case.in_dtype],
                                   code[case.out_dtype], s_i.cuda_stream)
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

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = _measured_peaks()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    achieved = case.flops / (per_launch_ms * 1e-3) / 1e12
    # 8-bit operands: no measured fp8 peak exists, so the measured bf16 figures
    # are scaled by the nominal dense fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s).
    # Packed 4-bit operands run on the same kind::mxf8f6f4 instruction as the
    # 8-bit ones (K = 32 per instruction), so their peak is the 8-bit one.
    rate = FP8_RATE if case.in_dtype in ("e4m3", "e5m2", "e2m1") else 1.0
    peak_burst = float(peaks["bf16_tflops"]) * rate
    peak_sustained = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * rate
    # The measured peaks come as a burst (a short cuBLAS run, clocks up) and a
    # sustained figure (seconds of back-to-back cuBLAS under the power cap).
    # The timed loop is held to the same condition as its denominator: a loop
    # that ran long enough to meet the power cap (>= 0.5 s, or sw_power_cap
    # seen while it ran) is compared with the sustained peak; a short loop, and
    # the burst figure, with the burst peak.
    power_capped = elapsed_ms >= 500.0 or bool(clocks and "sw_power_cap" in clocks.get("reasons", []))
    peak = peak_sustained if power_capped else peak_burst
    kind = "sustained" if power_capped else "burst"
    src = ("%s bf16 %s (cuBLAS 8192^3, MEASURED_PEAKS.json)%s; this loop: %d launches in %.0f ms%s" % (
        peak_src, kind, "; f16 runs at the bf16 rate" if rate == 1.0 else
        " x 2, the nominal dense fp8 / bf16 ratio", args.steps, elapsed_ms,
        ", sw_power_cap active" if clocks and "sw_power_cap" in clocks.get("reasons", []) else ""))
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
    roofline["burst"] = dict(burst, launches=BURST_STEPS, best_of=3, ms_per_launch=burst_ms)
    if case.mx:
        roofline["note"] = ("block-scaled: the time per launch is that of the whole gemm_mx step, the two small "
                            "scale-rearranging launches included" +
                            ("; packed E2M1 runs on kind::mxf8f6f4 at the 8-bit instruction rate, so the peak is "
                             "the 8-bit one" if case.in_dtype == "e2m1" else ""))
    if clocks and clocks.get("sm_mhz") and roofline["bound"] == "tensor":
        clk_peak = num_sms * FLOP_PER_CLK_PER_SM * rate * clocks["sm_mhz"] * 1e6 / 1e12
        roofline["frac_of_clock_peak"] = achieved / clk_peak
        roofline["clock_peak_tflops"] = clk_peak
    roofline["max_clock_peak_tflops"] = num_sms * FLOP_PER_CLK_PER_SM * rate * 2070e6 / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_launch_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": case.in_dtype, "data": "synthetic",
        "config": _workload_config(case, world), "roofline": roofline,
        "clocks": clocks, "e2e": e2e, "gpu_launches": args.steps * launches_per_step, "num_sms": num_sms,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = _args()
    from dense_tensor_core_02_gb300.inputs import CASE_BY_NAME, HEADLINE
    case = CASE_BY_NAME[args.case] if args.case else HEADLINE
    if args.impl == "reference":
        return run_reference(args, case)
    return run_ours(args, case)


if __name__ == "__main__":
    sys.exit(main())
