#!/usr/bin/env python3
"""Benchmark of the GB300 dense GEMM library.

Headline workload: half-precision GEMM C := 1.5*A*B + 0.5*C at M=N=K=4096
(fp16 operands, fp32 accumulation, fp16 C; A, B, C0 ~ U(-1,1) from the seeded
generator), reported as TFLOPS = 2MNK/t.  The fp32 SGEMM at 4096^3 (the other
half of the metric) is timed in the same run and reported beside it.

Timing (the method of the "advanced SGEMM on NVIDIA GPUs" page, benchmark
section): before every replay an L2-sized-or-larger buffer is cleared with
cudaMemsetAsync (outside the timed interval), then one CUDA-event pair on the
launching stream brackets the GEMM.  W untimed warm-up replays, then exactly K
timed ones; ms_per_step is the mean over the K replays (the page's "mean of
the second half" is reported too).  SM clocks are sampled with nvidia-smi
while the replays run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --sweep [--sweep-out FILE]    # fp32 size sweep 1024..12800
  python bench.py --sweep-f16 [--sweep-out FILE] [--sweep-sizes a,b,...]
                                                # fp16: automatic path vs the alternatives

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas, no collective on the data path); rank 0 prints the
line with value = total work of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("GEMM TFLOPS (2MNK/t) at 4096³ fp16-in/fp32-acc and fp32; "
          "% of tensor/FMA peak")
F16_CFG = dict(M=4096, N=4096, K=4096, alpha=1.5, beta=0.5)
PATH_FFMA_ONLY = 7          # gemm_force_path: the CUDA-core FFMA SGEMM only
F32_CFG = dict(M=4096, N=4096, K=4096, alpha=1.0, beta=0.0)
# (M, N, K, lda, alpha, beta, name): the fp16 edge shapes, ldb = ldc = N
EDGE_SHAPES = [
    (4097, 1023, 777, 780, 0.75, -0.25, "fp16 4097x1023x777, lda=780 (unaligned)"),
    (16, 8192, 8192, 8192, 0.75, -0.25, "fp16 skinny 16x8192x8192 (HBM-bound)"),
    (8192, 64, 4096, 4096, 0.75, -0.25, "fp16 tall 8192x64x4096 (HBM-bound)"),
]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SM_COUNT_NOMINAL = 152
FP32_LANES_PER_SM = 128


# ---------------------------------------------------------------- replay schedule

def replay_count(size: int) -> int:
    """Replays per size of the sweep: 1000*exp((1024 - size)/3100), truncated
    ("advanced SGEMM" page, benchmark section; 4096 -> 371)."""
    return int(1000.0 * math.exp((1024 - size) / 3100.0))


def second_half_mean(times):
    """Mean of the last floor(R/2) of R replay times (4096: the last 185 of 371)."""
    n = len(times) // 2
    tail = times[len(times) - n:] if n else times
    return sum(tail) / len(tail)


def sweep_sizes():
    return list(range(1024, 12800 + 1, 128))


# ---------------------------------------------------------------- helpers

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background (200 ms period)."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(prefix="clocks_", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.close()
        rows = []
        try:
            with open(self.out.name) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 10:
                        rows.append(parts)
        finally:
            os.unlink(self.out.name)
        return self._summary(rows)

    @staticmethod
    def _summary(rows):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        smax = [num(r[3]) for r in rows if num(r[3]) is not None]
        power = [num(r[4]) for r in rows if num(r[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {
            "sm_mhz": statistics.median(loaded) if loaded else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": reasons,
            "samples": len(rows),
            "power_w_max": max(power) if power else None,
        }


def _fill_device(shape, dtype_np, seed, stream_id, dist="uniform"):
    import torch
    import synthetic
    gen = synthetic.uniform if dist == "uniform" else synthetic.normal
    host = gen(seed, stream_id, shape, dtype=dtype_np)
    return torch.from_numpy(host).cuda(), host


# ---------------------------------------------------------------- ranks

def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of `values` (a list of floats) over all ranks of
    the default process group: the slowest rank's times decide the job's
    throughput.  `device` is where the reduction runs ("cuda" under NCCL,
    "cpu" under gloo)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


# ---------------------------------------------------------------- device-timed replays

class LaunchTally:
    """Kernels the library launched inside timed regions (its own counter,
    read before and after each region)."""
    total = 0


def timed_replays(fn, steps, warmup, stream, flush_bytes):
    """W warm-up + K timed replays; L2 flush before each, one event pair per
    replay on `stream`.  Returns per-replay milliseconds; the library's
    launches during the K timed replays are added to LaunchTally."""
    import torch
    import dense_gemm_03_gb300 as g
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.l2_flush(flush_bytes, stream)
            fn()
        torch.cuda.synchronize()
        n0 = g.launch_count()
        for i in range(steps):
            g.l2_flush(flush_bytes, stream)
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
        torch.cuda.synchronize()
        LaunchTally.last = g.launch_count() - n0
        LaunchTally.total += LaunchTally.last
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def run_ours(args, rank, world):
    import torch
    import dense_gemm_03_gb300 as g
    import synthetic
    from dense_gemm_03_gb300 import build as _b

    _b.build()
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    flush_bytes = 2 * l2
    peaks, peaks_src = _peaks()

    # fp16 headline workload
    M, N, K = F16_CFG["M"], F16_CFG["N"], F16_CFG["K"]
    seed = synthetic.config_seed(2)
    dA, hA = _fill_device((M, K), np.float16, seed, synthetic.STREAM_A)
    dB, hB = _fill_device((K, N), np.float16, seed, synthetic.STREAM_B)
    dC, hC = _fill_device((M, N), np.float16, seed, synthetic.STREAM_C)
    f16 = lambda: g.gemm_f16(dA, dB, dC, F16_CFG["alpha"], F16_CFG["beta"], stream=stream)

    # fp32 workload
    seed32 = synthetic.config_seed(1)
    fA, _ = _fill_device((M, K), np.float32, seed32, synthetic.STREAM_A)
    fB, _ = _fill_device((K, N), np.float32, seed32, synthetic.STREAM_B)
    fC = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    f32 = lambda: g.sgemm_f32(fA, fB, fC, 1.0, 0.0, stream=stream)

    peak16_local = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(dev).start()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    ms16 = timed_replays(f16, args.steps, args.warmup, stream, flush_bytes)
    path16 = g.last_path()
    launches16 = LaunchTally.last / args.steps
    f32_steps = max(3, args.steps // 20)
    prev_path = g.force_path(PATH_FFMA_ONLY) if args.f32_ffma else None
    ms32 = timed_replays(f32, f32_steps, max(3, args.warmup // 10), stream, flush_bytes)
    path32 = g.last_path()
    if prev_path is not None:
        g.force_path(prev_path)
    launches32 = LaunchTally.last / f32_steps
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    clocks = sampler.stop()
    assert g.debug_status() == 0, "a kernel reported a timeout"

    mean16 = sum(ms16) / len(ms16)
    mean32 = sum(ms32) / len(ms32)
    if world > 1:
        mean16, mean32 = max_over_ranks([mean16, mean32], device="cuda")
    flops = 2.0 * M * N * K
    tflops16 = flops / (mean16 * 1e-3) / 1e12
    tflops32 = flops / (mean32 * 1e-3) / 1e12

    # fp16 operands with an fp32 C, and the fp32 -> fp16 conversion of C
    f32c = torch.from_numpy(synthetic.uniform(seed, synthetic.STREAM_C, (M, N),
                                              dtype=np.float32)).cuda()
    fo = lambda: g.gemm_f16_f32out(dA, dB, f32c, F16_CFG["alpha"], F16_CFG["beta"], stream=stream)
    ms_fo = timed_replays(fo, max(20, args.steps // 20), 5, stream, flush_bytes)
    path_fo = g.last_path()
    conv_dst = torch.empty((M, N), dtype=torch.float16, device="cuda")
    cv = lambda: g.f32_to_f16(f32c, conv_dst, stream=stream)
    ms_cv = timed_replays(cv, max(20, args.steps // 20), 5, stream, flush_bytes)
    t_fo = sum(ms_fo) / len(ms_fo)
    t_cv = sum(ms_cv) / len(ms_cv)
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    extra = {
        "f16_f32out": {
            "workload": "fp16 A, B -> fp32 C = 1.5*A*B + 0.5*C, M=N=K=4096",
            "us": round(t_fo * 1e3, 2),
            "tflops": round(2.0 * M * N * K / (t_fo * 1e-3) / 1e12, 1),
            "frac_tensor": round(2.0 * M * N * K / (t_fo * 1e-3) / 1e12 / peak16_local, 4),
            "kernel_path": path_fo,
        },
        "f32_to_f16": {
            "workload": "fp32 -> fp16 conversion of a 4096 x 4096 matrix",
            "us": round(t_cv * 1e3, 2),
            "gb_s": round(6.0 * M * N / (t_cv * 1e-3) / 1e9, 1),
            "frac_hbm": round(6.0 * M * N / (t_cv * 1e-3) / 1e9 / hbm_peak, 4),
            "algorithmic_bytes": 6 * M * N,
        },
    }
    del f32c, conv_dst

    # the other workloads of the metric, timed the same way (context for the headline)
    shapes = []
    squares = []
    if not args.no_shapes:
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        for (sM, sN, sK, slda, alpha, beta, name) in EDGE_SHAPES:
            seed_e = synthetic.config_seed(4)
            eA, _ = _fill_device((sM * slda,), np.float16, seed_e, synthetic.STREAM_A)
            eB, _ = _fill_device((sK, sN), np.float16, seed_e, synthetic.STREAM_B)
            eC, _ = _fill_device((sM, sN), np.float16, seed_e, synthetic.STREAM_C)
            fn = lambda: g.gemm_f16(eA, eB, eC, alpha, beta, M=sM, N=sN, K=sK, lda=slda, ldb=sN,
                                    ldc=sN, stream=stream)
            ms = timed_replays(fn, max(20, args.steps // 20), 5, stream, flush_bytes)
            t = sum(ms) / len(ms)
            byts = 2 * (sM * sK + sK * sN) + 2 * 2 * sM * sN
            fl = 2.0 * sM * sN * sK
            tf = fl / (t * 1e-3) / 1e12
            gbs = byts / (t * 1e-3) / 1e9
            shapes.append({"workload": name, "us": round(t * 1e3, 2), "tflops": round(tf, 1),
                           "gb_s": round(gbs, 1), "frac_tensor": round(tf / peak16_local, 3),
                           "frac_hbm": round(gbs / hbm, 3), "kernel_path": g.last_path()})
            del eA, eB, eC
        # the fp32 square configurations below 4096 (4096 is the fp32 leg above)
        ceiling32 = peak16_local * (1.1 / 2.25) / 3.0
        for n in (256, 512, 1024, 2048):
            seed_s = synthetic.config_seed(1)
            sA, _ = _fill_device((n, n), np.float32, seed_s, synthetic.STREAM_A)
            sB, _ = _fill_device((n, n), np.float32, seed_s, synthetic.STREAM_B)
            sC = torch.zeros((n, n), dtype=torch.float32, device="cuda")
            fn = lambda: g.sgemm_f32(sA, sB, sC, 1.0, 0.0, stream=stream)
            ms = timed_replays(fn, max(20, args.steps // 20), 5, stream, flush_bytes)
            t = sum(ms) / len(ms)
            tf = 2.0 * n ** 3 / (t * 1e-3) / 1e12
            squares.append({"workload": "fp32 SGEMM %d^3, alpha=1 beta=0" % n,
                            "us": round(t * 1e3, 2), "tflops": round(tf, 2),
                            "frac_3xtf32_ceiling": round(tf / ceiling32, 4),
                            "kernel_path": g.last_path()})
            del sA, sB, sC

    # end to end through the host-buffer C-ABI call (copies inside the timed region)
    pA = torch.from_numpy(hA).pin_memory()
    pB = torch.from_numpy(hB).pin_memory()
    pC = torch.from_numpy(hC.copy()).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        g.gemm_f16_host(pA, pB, pC, F16_CFG["alpha"], F16_CFG["beta"], stream=stream)
    e2e_ms = []
    n0 = g.launch_count()
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        g.gemm_f16_host(pA, pB, pC, F16_CFG["alpha"], F16_CFG["beta"], stream=stream)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    LaunchTally.total += g.launch_count() - n0
    e2e_mean = sum(e2e_ms) / len(e2e_ms)
    if world > 1:
        (e2e_mean,) = max_over_ranks([e2e_mean], device="cuda")

    peak16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    sm_count = props.multi_processor_count or SM_COUNT_NOMINAL
    peak_ffma = sm_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    traffic = _profiled_traffic("tc_f16_4096")
    if path32.startswith("f32.3xtf32"):
        # three tf32 tensor products per fp32 multiply-add: the fp32 ceiling is
        # a third of the tf32 dense rate (the bf16 peak x the nominal
        # tf32/bf16 ratio of 1.1/2.25 PFLOP/s)
        peak32 = peak16 * (1.1 / 2.25) / 3.0
        roof32 = {"bound": "tensor", "achieved": round(tflops32, 2), "peak": round(peak32, 2),
                  "unit": "TFLOP/s", "frac": round(tflops32 / peak32, 4),
                  "traffic": _profiled_traffic("sgemm_3xtf32_4096"),
                  "peak_source": "%s bf16 dense burst x 1.1/2.25 (tf32 nominal ratio) / 3 tf32 "
                                 "products per fp32 FLOP" % peaks_src,
                  "launches_per_step": launches32,
                  "note": "time includes the operand-split pre-passes",
                  "vs_ffma_peak": round(tflops32 / peak_ffma, 3)}
    else:
        peak32 = peak_ffma
        roof32 = {"bound": "alu", "achieved": round(tflops32, 2), "peak": round(peak32, 2),
                  "unit": "TFLOP/s", "frac": round(tflops32 / peak32, 4),
                  "traffic": _profiled_traffic("sgemm_ffma_4096"),
                  "peak_source": "%d SMs x 128 FP32 lanes x 2 FLOP x %.0f MHz" % (sm_count, sm_max),
                  "launches_per_step": launches32}

    line = {
        "metric": METRIC,
        "value": round(tflops16 * world, 3),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean16, 6),
        "ms_per_step_second_half": round(second_half_mean(ms16), 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded splitmix64, U(-1,1) rounded to fp16)",
        "config": {
            "workload": "fp16 GEMM C=1.5*A*B+0.5*C, M=N=K=4096, row-major, fp32 accumulate",
            "M": M, "N": N, "K": K, "alpha": F16_CFG["alpha"], "beta": F16_CFG["beta"],
            "l2": "flushed before every replay (cudaMemsetAsync of %d MiB)" % (flush_bytes >> 20),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "kernel_path": path16,
        },
        "roofline": {
            "bound": "tensor",
            "achieved": round(tflops16, 2),
            "peak": peak16,
            "unit": "TFLOP/s",
            "frac": round(tflops16 / peak16, 4),
            "peak_source": "%s bf16 dense burst (fp16 dense has the same rate)" % peaks_src,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": 2 * (M * K + K * N) + 2 * 2 * M * N,
            "launches_per_step": launches16,
        },
        "fp32_sgemm": {
            "workload": "fp32 SGEMM C=A*B, M=N=K=4096, alpha=1 beta=0" +
                        (" (CUDA-core FFMA kernel forced)" if args.f32_ffma else ""),
            "value": round(tflops32 * world, 3),
            "unit": "TFLOPS",
            "ms_per_step": round(mean32, 5),
            "steps": f32_steps,
            "kernel_path": path32,
            "roofline": roof32,
            "context_vs_page_colab_86ms": round(tflops32 / (2 * 4096 ** 3 / 86.1e-3 / 1e12), 1),
        },
        "e2e": {
            "value": round(flops * world / (e2e_mean * 1e-3) / 1e12, 3),
            "unit": "TFLOPS",
            "h2d_bytes_per_step": int(hA.nbytes + hB.nbytes + hC.nbytes),
            "d2h_bytes_per_step": int(hC.nbytes),
            "ms_per_step": round(e2e_mean, 4),
            "api": "gemm_f16_host (pinned host buffers)",
        },
        "edge_shapes": shapes,
        "fp32_squares": squares,
        **extra,
        "gpu_launches": LaunchTally.total,
        "clocks": clocks,
        "wall_s_timed": round(t_wall1 - t_wall0, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


def _profiled_traffic(key):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    (profiles/traffic.json), or None when there is none or when the kernel's
    sources changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(key)
        if not rec:
            return None
        h = hashlib.sha1()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        return rec["dram_bytes_per_launch"] if h.hexdigest() == rec["sources_sha1"] else None
    except (OSError, ValueError, KeyError):
        return None


# ---------------------------------------------------------------- CPU oracle legs

def cpu_baseline(seconds: float):
    """The oracle (plain triple loop in double) on a bounded sample of the
    headline workload: as many full rows of C as fit in about `seconds`."""
    import oracle
    import synthetic
    M, N, K = F16_CFG["M"], F16_CFG["N"], F16_CFG["K"]
    seed = synthetic.config_seed(2)
    A = synthetic.uniform(seed, synthetic.STREAM_A, (M, K), dtype=np.float16)
    B = synthetic.uniform(seed, synthetic.STREAM_B, (K, N), dtype=np.float16)
    C0 = synthetic.uniform(seed, synthetic.STREAM_C, (M, N), dtype=np.float16)
    cores = oracle.max_threads()
    rows = max(cores, 8)
    t = _time_rows(oracle, A, B, C0, rows)
    target_rows = int(min(M, max(rows, rows * seconds / max(t, 1e-6))))
    t = _time_rows(oracle, A, B, C0, target_rows)
    flops = 2.0 * target_rows * N * K
    # the oracle on one thread, on the two smallest fp32 workloads (256^3, 1024^3)
    single = {}
    oracle.set_threads(1)
    try:
        for n in (256, 1024):
            sa = synthetic.uniform(synthetic.config_seed(1), synthetic.STREAM_A, (n, n))
            sb = synthetic.uniform(synthetic.config_seed(1), synthetic.STREAM_B, (n, n))
            t0 = time.perf_counter()
            oracle.gemm(sa, sb, None, 1.0, 0.0)
            dt = time.perf_counter() - t0
            single["fp32 %d^3" % n] = {"s": round(dt, 4), "tflops": round(2.0 * n ** 3 / dt / 1e12, 6)}
    finally:
        oracle.set_threads(cores)
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOPS", "cores": cores,
            "kind": "oracle",
            "sample": "%d of %d rows of C for the fp16 4096^3 workload (%.1f s)" % (target_rows, M, t),
            "single_thread": single}


def _time_rows(oracle, A, B, C0, nrows):
    rows = list(range(nrows))
    t0 = time.perf_counter()
    oracle.gemm(A, B, C0, F16_CFG["alpha"], F16_CFG["beta"], rows=rows)
    return time.perf_counter() - t0


def run_reference(args):
    """Reference arm: the CPU oracle on the machine's host cores, timed on a
    bounded sample of the same workload each step."""
    import oracle
    import synthetic
    M, N, K = F16_CFG["M"], F16_CFG["N"], F16_CFG["K"]
    seed = synthetic.config_seed(2)
    A = synthetic.uniform(seed, synthetic.STREAM_A, (M, K), dtype=np.float16)
    B = synthetic.uniform(seed, synthetic.STREAM_B, (K, N), dtype=np.float16)
    C0 = synthetic.uniform(seed, synthetic.STREAM_C, (M, N), dtype=np.float16)
    cores = oracle.max_threads()
    rows_per_step = max(cores, 8)
    budget = 120.0 / max(1, args.steps + args.warmup)     # whole run within ~2 minutes
    t = _time_rows(oracle, A, B, C0, rows_per_step)
    rows_per_step = int(min(M, max(1, rows_per_step * min(budget, 5.0) / max(t, 1e-6))))
    for _ in range(args.warmup):
        _time_rows(oracle, A, B, C0, rows_per_step)
    times = [_time_rows(oracle, A, B, C0, rows_per_step) for _ in range(args.steps)]
    mean = sum(times) / len(times)
    flops = 2.0 * rows_per_step * N * K
    value = flops / mean / 1e12
    sample = "%d of %d rows of C per step for the fp16 4096^3 workload" % (rows_per_step, M)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded splitmix64)",
        "config": {"workload": "fp16 GEMM C=1.5*A*B+0.5*C, M=N=K=4096, row-major (CPU oracle, "
                               "sampled rows)", "M": M, "N": N, "K": K},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- fp32 sweep

def run_sweep(args):
    import torch
    import dense_gemm_03_gb300 as g
    import synthetic
    from dense_gemm_03_gb300 import build as _b
    _b.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(0)
    flush = 2 * int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    out = open(args.sweep_out, "a") if args.sweep_out else None
    done = set()
    if args.sweep_out and os.path.exists(args.sweep_out):
        with open(args.sweep_out) as f:
            for line in f:
                try:
                    done.add(json.loads(line)["size"])
                except (ValueError, KeyError):
                    pass
    sizes = [s for s in sweep_sizes() if s not in done]
    if args.sweep_sizes:
        sizes = [int(x) for x in args.sweep_sizes.split(",")]
    sampler = ClockSampler(0).start()
    results = []
    for n in sizes:
        seed = synthetic.config_seed(3) + n
        A = torch.from_numpy(synthetic.normal(seed, synthetic.STREAM_A, (n, n))).cuda()
        B = torch.from_numpy(synthetic.normal(seed, synthetic.STREAM_B, (n, n))).cuda()
        C = torch.zeros((n, n), dtype=torch.float32, device="cuda")
        R = replay_count(n)
        ms = timed_replays(lambda: g.sgemm_f32(A, B, C, 1.0, 0.0, stream=stream), R, 0, stream, flush)
        t = second_half_mean(ms)
        rec = {"size": n, "replays": R, "ms_second_half_mean": round(t, 5),
               "tflops": round(2.0 * n ** 3 / (t * 1e-3) / 1e12, 3), "kernel_path": g.last_path()}
        results.append(rec)
        if out:
            out.write(json.dumps(rec) + "\n")
            out.flush()
        del A, B, C
    clocks = sampler.stop()
    print(json.dumps({"sweep": "fp32 SGEMM 1024..12800 step 128", "sizes": len(results),
                      "clocks": clocks,
                      "tflops_mean": round(sum(r["tflops"] for r in results) / max(1, len(results)), 3)}))


# ---------------------------------------------------------------- fp16 tile-heuristic sweep

F16_VARIANTS = [(0, "auto"), (6, "no_pairs"), (5, "whole_tiles"), (9, "k_slices_tail"),
                (10, "stream_k")]


def run_sweep_f16(args):
    """Square fp16 GEMMs (C = 1.5*A*B + 0.5*C) over the sweep sizes: the
    automatic path and the forced alternatives it chooses between, each timed
    the same way (L2 cleared before every replay, second-half mean of a
    quarter of the page's replay count)."""
    import torch
    import dense_gemm_03_gb300 as g
    import synthetic
    from dense_gemm_03_gb300 import build as _b
    _b.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(0)
    flush = 2 * int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    out = open(args.sweep_out, "a") if args.sweep_out else None
    sizes = sweep_sizes()
    if args.sweep_sizes:
        sizes = [int(x) for x in args.sweep_sizes.split(",")]
    sampler = ClockSampler(0).start()
    best_is_auto = 0
    within = 0
    for n in sizes:
        seed = synthetic.config_seed(5) + n
        A = torch.from_numpy(synthetic.uniform(seed, synthetic.STREAM_A, (n, n), dtype=np.float16)).cuda()
        B = torch.from_numpy(synthetic.uniform(seed, synthetic.STREAM_B, (n, n), dtype=np.float16)).cuda()
        C = torch.from_numpy(synthetic.uniform(seed, synthetic.STREAM_C, (n, n), dtype=np.float16)).cuda()
        R = max(8, replay_count(n) // 4)
        rec = {"size": n, "replays": R}
        for path, name in F16_VARIANTS:
            prev = g.force_path(path)
            try:
                ms = timed_replays(lambda: g.gemm_f16(A, B, C, 1.5, 0.5, stream=stream), R, 3,
                                   stream, flush)
                rec[name] = {"us": round(second_half_mean(ms) * 1e3, 2), "path": g.last_path()}
            finally:
                g.force_path(prev)
        rec["tflops_auto"] = round(2.0 * n ** 3 / (rec["auto"]["us"] * 1e-6) / 1e12, 1)
        best = min(v["us"] for k, v in rec.items() if isinstance(v, dict))
        rec["auto_vs_best"] = round(rec["auto"]["us"] / best, 4)
        best_is_auto += rec["auto"]["us"] <= best
        within += rec["auto_vs_best"] <= 1.02
        if out:
            out.write(json.dumps(rec) + "\n")
            out.flush()
        del A, B, C
    clocks = sampler.stop()
    print(json.dumps({"sweep": "fp16 heuristic 1024..12800 step 128", "sizes": len(sizes),
                      "auto_best": best_is_auto, "auto_within_2pct": within, "clocks": clocks}))


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-shapes", action="store_true", help="skip the edge-shape timings")
    ap.add_argument("--f32-ffma", action="store_true",
                    help="time the fp32 leg on the CUDA-core FFMA kernel instead of 3xTF32")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-f16", action="store_true",
                    help="fp16 sweep: the automatic path beside the forced alternatives")
    ap.add_argument("--sweep-out", default=None)
    ap.add_argument("--sweep-sizes", default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.sweep_f16:
        run_sweep_f16(args)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
