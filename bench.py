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
  python bench.py --sweep-tall [--sweep-out FILE]
                                                # fp16 tall shapes (N <= 64): schedules

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
    """SM clock, clock-event (throttle) reasons and power, sampled through NVML
    (libnvidia-ml, read-only queries) every `period` seconds by a background
    thread.  `mark(name)` / `end(name)` bracket host-time windows (a timed
    region: from the first enqueue to the synchronise after the last replay);
    `summary(names)` summarises the samples that fall inside those windows.
    Without NVML it falls back to nvidia-smi at its 100 ms minimum period."""

    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    IDLE_BIT = 0x1

    def __init__(self, cuda_index: int, period: float = 0.002):
        self.period = period
        self.samples = []          # (t, sm_mhz, max_mhz, reasons, power_w)
        self.windows = {}
        self._stop = None
        self._thread = None
        self._smi = None
        self.source = "none"
        self._nvml = self._open_nvml(cuda_index)

    @staticmethod
    def _open_nvml(cuda_index):
        import ctypes
        try:
            L = ctypes.CDLL("libnvidia-ml.so.1")
            if L.nvmlInit_v2() != 0:
                return None
        except OSError:
            return None
        h = ctypes.c_void_p()
        found = False
        try:
            import torch
            props = torch.cuda.get_device_properties(cuda_index)
            uuid = str(getattr(props, "uuid", "") or "")
            if uuid:
                key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                found = L.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(h)) == 0
            if not found and hasattr(props, "pci_bus_id"):
                bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id,
                                            props.pci_device_id)
                found = L.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
        except Exception:
            found = False
        if not found and L.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(h)) != 0:
            return None
        reasons = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(L, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        return (L, h, reasons)

    def _sample_nvml(self):
        import ctypes
        L, h, reasons_fn = self._nvml
        clk, mx, pw = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_uint(0)
        rs = ctypes.c_ulonglong(0)
        t = time.perf_counter()
        ok = L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0      # NVML_CLOCK_SM
        L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        if reasons_fn is not None:
            reasons_fn(h, ctypes.byref(rs))
        L.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
        if ok:
            self.samples.append((t, float(clk.value), float(mx.value), int(rs.value),
                                 pw.value / 1000.0))

    def start(self):
        import threading
        if self._nvml is not None:
            self.source = "nvml, %.0f ms period" % (self.period * 1e3)
            self._stop = threading.Event()

            def loop():
                while not self._stop.is_set():
                    try:
                        self._sample_nvml()
                    except Exception:
                        return
                    time.sleep(self.period)
            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
        else:
            self.source = "nvidia-smi, 100 ms period"
            self._t0 = time.perf_counter()
            self._smi_out = tempfile.NamedTemporaryFile(prefix="clocks_", suffix=".csv",
                                                        delete=False)
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=timestamp,clocks.sm,clocks.max.sm,power.draw,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=self._smi_out, stderr=subprocess.DEVNULL)
            except OSError:
                self._smi = None
        return self

    def mark(self, name):
        self.windows[name] = [time.perf_counter(), None]

    def end(self, name):
        self.windows[name][1] = time.perf_counter()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self._smi is not None:
            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
            self._smi_out.close()
            # nvidia-smi rows carry no perf_counter time: spread them evenly
            rows = []
            with open(self._smi_out.name) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 5:
                        rows.append(parts)
            os.unlink(self._smi_out.name)
            t1 = time.perf_counter()
            for i, r in enumerate(rows):
                try:
                    t = self._t0 + (t1 - self._t0) * (i + 0.5) / len(rows)
                    self.samples.append((t, float(r[1]), float(r[2]), int(r[4], 16),
                                         float(r[3])))
                except ValueError:
                    pass
        return self

    def summary(self, names=None):
        """Samples inside the named windows (all samples when names is None)."""
        if names is None:
            sel = list(self.samples)
        else:
            wins = [self.windows[n] for n in names if n in self.windows and self.windows[n][1]]
            sel = [x for x in self.samples if any(a <= x[0] <= b for a, b in wins)]
        smax = max((x[2] for x in sel), default=None)
        loaded = [x for x in sel if not (x[3] & self.IDLE_BIT) and
                  (smax is None or x[1] > 0.5 * smax)]
        reasons = sorted({name for x in loaded for bit, name in self.REASON_BITS.items()
                          if x[3] & bit})
        return {
            "sm_mhz": statistics.median([x[1] for x in loaded]) if loaded else None,
            "sm_max_mhz": smax,
            "reasons": reasons,
            "samples": len(sel),
            "samples_under_load": len(loaded),
            "power_w_max": max((x[4] for x in sel), default=None),
            "source": self.source,
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


def timed_replays(fn, steps, warmup, stream, flush_bytes, sampler=None, window=None):
    """W warm-up + K timed replays; L2 flush before each, one event pair per
    replay on `stream`.  Returns per-replay milliseconds; the library's
    launches during the K timed replays are added to LaunchTally.  With a
    sampler, the timed replays form the clock window `window`."""
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
        if sampler is not None:
            sampler.mark(window)
        for i in range(steps):
            g.l2_flush(flush_bytes, stream)
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
        torch.cuda.synchronize()
        if sampler is not None:
            sampler.end(window)
        LaunchTally.last = g.launch_count() - n0
        LaunchTally.total += LaunchTally.last
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def sustained_replays(fn, seconds, stream, flush_bytes, sampler, window, batch=200):
    """The same replays (flush, event pair, call) back to back for about
    `seconds` of wall time, in batches; returns per-replay milliseconds."""
    import torch
    import dense_gemm_03_gb300 as g
    out = []
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(batch)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(batch)]
    n0 = g.launch_count()
    sampler.mark(window)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        while time.perf_counter() - t0 < seconds:
            for i in range(batch):
                g.l2_flush(flush_bytes, stream)
                starts[i].record(stream)
                fn()
                ends[i].record(stream)
            torch.cuda.synchronize()
            out.extend(s.elapsed_time(e) for s, e in zip(starts, ends))
    sampler.end(window)
    LaunchTally.total += g.launch_count() - n0
    return out


def measured_tf32_tflops(n=8192, reps=10):
    """Dense tf32 rate of this GPU, measured off the library's path like the
    bf16 figure of the peaks file: torch.matmul on fp32 operands with tf32
    allowed (cuBLAS), n^3, best of `reps` after 3 warm-ups, CUDA events."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        gen = torch.Generator(device="cuda").manual_seed(1)
        a = torch.randn((n, n), device="cuda", generator=gen)
        b = torch.randn((n, n), device="cuda", generator=gen)
        c = torch.empty((n, n), device="cuda")
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b, c
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


# fp32 size-sweep sizes timed in the default line: every eighth size of the
# 1024..12800 step-128 sweep, and its last one
SWEEP_SUBSET = list(range(1024, 12800, 1024)) + [12800]


def sweep_subset(stream, flush_bytes, sampler, sizes=SWEEP_SUBSET):
    """The fp32 sweep's schedule (R(n) replays, L2 flushed before each,
    second-half mean) on a subset of its sizes.  Operands: N(0,1) filled on
    the device by a seeded torch generator (timing only; the parity tests use
    the host generator)."""
    import torch
    import dense_gemm_03_gb300 as g
    gen = torch.Generator(device="cuda").manual_seed(3)
    nmax = max(sizes)
    A = torch.randn((nmax * nmax,), device="cuda", generator=gen)
    B = torch.randn((nmax * nmax,), device="cuda", generator=gen)
    C = torch.zeros((nmax * nmax,), device="cuda")
    res = []
    sampler.mark("fp32_sweep")
    for n in sizes:
        a, b, c = A[:n * n], B[:n * n], C[:n * n]
        R = replay_count(n)
        ms = timed_replays(lambda: g.sgemm_f32(a, b, c, 1.0, 0.0, M=n, N=n, K=n, stream=stream),
                           R, 3, stream, flush_bytes)
        t = second_half_mean(ms)
        res.append({"n": n, "replays": R, "tflops": round(2.0 * n ** 3 / (t * 1e-3) / 1e12, 1)})
    sampler.end("fp32_sweep")
    del A, B, C
    tf = [r["tflops"] for r in res]
    return {"workload": "fp32 SGEMM m=n=k sweep subset (every 8th size of 1024..12800 step 128, "
                        "and 12800), R(n) = 1000*exp((1024-n)/3100) replays, second-half mean",
            "kernel_path": g.last_path(), "tflops_mean": round(sum(tf) / len(tf), 1),
            "tflops_min": min(tf), "tflops_max": max(tf), "sizes": res}


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
    sm_count = props.multi_processor_count or SM_COUNT_NOMINAL
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))

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
    ms16 = timed_replays(f16, args.steps, args.warmup, stream, flush_bytes, sampler, "fp16")
    path16 = g.last_path()
    launches16 = LaunchTally.last / args.steps
    t_wall1 = time.perf_counter()
    # the headline replays again, back to back for a few seconds: enough clock
    # samples under load, and the rate once power limits have settled
    ms16s = sustained_replays(f16, args.sustain_seconds, stream, flush_bytes, sampler,
                              "fp16_sustained") if args.sustain_seconds > 0 else []
    f32_steps = max(50, args.steps // 20)
    prev_path = g.force_path(PATH_FFMA_ONLY) if args.f32_ffma else None
    ms32 = timed_replays(f32, f32_steps, 5, stream, flush_bytes, sampler, "fp32")
    path32 = g.last_path()
    if prev_path is not None:
        g.force_path(prev_path)
    launches32 = LaunchTally.last / f32_steps
    # the CUDA-core FFMA SGEMM on the same workload (forced)
    prev_path = g.force_path(PATH_FFMA_ONLY)
    try:
        ms_ffma = timed_replays(f32, 20, 3, stream, flush_bytes, sampler, "fp32_ffma")
        path_ffma = g.last_path()
    finally:
        g.force_path(prev_path)
    torch.cuda.synchronize()
    assert g.debug_status() == 0, "a kernel reported a timeout"

    mean16 = sum(ms16) / len(ms16)
    mean32 = sum(ms32) / len(ms32)
    mean_ffma = sum(ms_ffma) / len(ms_ffma)
    if world > 1:
        mean16, mean32 = max_over_ranks([mean16, mean32], device="cuda")
    flops = 2.0 * M * N * K
    tflops16 = flops / (mean16 * 1e-3) / 1e12
    tflops32 = flops / (mean32 * 1e-3) / 1e12
    tflops_ffma = flops / (mean_ffma * 1e-3) / 1e12

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
    sweep = None
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
        # the fp32 square configurations below 4096 (4096 is the fp32 leg
        # above); each one's fraction of its own kernel's ceiling is added
        # once the tf32 rate has been measured
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
                            "kernel_path": g.last_path()})
            del sA, sB, sC
        del fA, fB, fC
        sweep = sweep_subset(stream, flush_bytes, sampler)

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

    tf32_meas = None
    if not args.no_tf32_peak:
        try:
            tf32_meas = measured_tf32_tflops()
        except Exception:        # noqa: BLE001 -- the denominator falls back to the nominal ratio
            tf32_meas = None
    sampler.stop()
    clk16 = sampler.summary(["fp16", "fp16_sustained"])
    clk32 = sampler.summary(["fp32"])
    clk_ffma = sampler.summary(["fp32_ffma"])

    peak16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_ffma = sm_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    traffic = _profiled_traffic("tc_f16_4096")
    # ceilings of the two split-operand fp32 kernels: three tensor products per
    # fp32 multiply-add, so a third of the dense fp16 rate (3xFP16; the
    # measured bf16 burst, the same tensor rate) or of the dense tf32 rate
    # (3xTF32: measured in this run when possible, else the bf16 peak x the
    # nominal tf32/bf16 ratio 1.1/2.25)
    ceil_f16x3 = peak16 / 3.0
    nominal32 = peak16 * (1.1 / 2.25) / 3.0
    ceil_tf32x3 = tf32_meas / 3.0 if tf32_meas else nominal32
    for sq in squares:
        c = ceil_f16x3 if sq["kernel_path"].startswith("f32.3xf16") else (
            ceil_tf32x3 if sq["kernel_path"].startswith("f32.3xtf32") else None)
        sq["frac_ceiling"] = round(sq["tflops"] / c, 4) if c else None
    if path32.startswith("f32.3xf16"):
        peak32 = ceil_f16x3
        roof32 = {"bound": "tensor", "achieved": round(tflops32, 2), "peak": round(peak32, 2),
                  "unit": "TFLOP/s", "frac": round(tflops32 / peak32, 4),
                  "traffic": _profiled_traffic("sgemm_3xf16_4096"),
                  "peak_source": ("%s bf16 dense burst (the same tensor rate as fp16) / 3 fp16 "
                                  "products per fp32 FLOP" % peaks_src),
                  "launches_per_step": launches32,
                  "note": "time includes the operand-split pre-passes",
                  "vs_ffma_peak": round(tflops32 / peak_ffma, 3)}
    elif path32.startswith("f32.3xtf32"):
        if tf32_meas:
            peak32 = tf32_meas / 3.0
            src32 = ("dense tf32 rate measured in this run (torch.matmul fp32 with tf32 allowed, "
                     "8192^3, best of 10: %.1f TFLOP/s) / 3 tf32 products per fp32 FLOP" % tf32_meas)
        else:
            peak32 = nominal32
            src32 = ("%s bf16 dense burst x 1.1/2.25 (tf32 nominal ratio) / 3 tf32 products per "
                     "fp32 FLOP" % peaks_src)
        roof32 = {"bound": "tensor", "achieved": round(tflops32, 2), "peak": round(peak32, 2),
                  "unit": "TFLOP/s", "frac": round(tflops32 / peak32, 4),
                  "traffic": _profiled_traffic("sgemm_3xtf32_4096"),
                  "peak_source": src32, "frac_of_nominal_ratio_ceiling": round(tflops32 / nominal32, 4),
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
    ffma_clock_peak = (sm_count * FP32_LANES_PER_SM * 2 * clk_ffma["sm_mhz"] * 1e6 / 1e12
                       if clk_ffma["sm_mhz"] else None)
    mean16s = sum(ms16s) / len(ms16s) if ms16s else None

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
        "fp16_sustained": {
            "workload": "the headline replays (flush, event pair, GEMM) back to back for %.1f s"
                        % args.sustain_seconds,
            "replays": len(ms16s),
            "us": round(mean16s * 1e3, 2) if mean16s else None,
            "tflops": round(flops / (mean16s * 1e-3) / 1e12, 1) if mean16s else None,
            "frac": round(flops / (mean16s * 1e-3) / 1e12 / peak16, 4) if mean16s else None,
            "clocks": sampler.summary(["fp16_sustained"]),
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
            "clocks": clk32,
            "context_vs_page_colab_86ms": round(tflops32 / (2 * 4096 ** 3 / 86.1e-3 / 1e12), 1),
        },
        "fp32_ffma": {
            "workload": "fp32 SGEMM C=A*B, M=N=K=4096, alpha=1 beta=0, CUDA-core FFMA kernel forced",
            "tflops": round(tflops_ffma, 2),
            "ms_per_step": round(mean_ffma, 4),
            "steps": len(ms_ffma),
            "kernel_path": path_ffma,
            "roofline": {"bound": "alu", "achieved": round(tflops_ffma, 2),
                         "peak": round(peak_ffma, 2), "unit": "TFLOP/s",
                         "frac": round(tflops_ffma / peak_ffma, 4),
                         "peak_source": "%d SMs x 128 FP32 lanes x 2 FLOP x %.0f MHz (max clock)"
                                        % (sm_count, sm_max),
                         "frac_at_sampled_clock": (round(tflops_ffma / ffma_clock_peak, 4)
                                                   if ffma_clock_peak else None),
                         "traffic": _profiled_traffic("sgemm_ffma_4096")},
            "clocks": clk_ffma,
        },
        "fp32_sweep": sweep,
        "tf32_dense_tflops_measured": round(tf32_meas, 1) if tf32_meas else None,
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
        "clocks": clk16,
        "clock_scaled_ms": (round(mean16 * clk16["sm_mhz"], 3) if clk16["sm_mhz"] else None),
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
    clocks = sampler.stop().summary()
    print(json.dumps({"sweep": "fp32 SGEMM 1024..12800 step 128", "sizes": len(results),
                      "clocks": clocks,
                      "tflops_mean": round(sum(r["tflops"] for r in results) / max(1, len(results)), 3)}))


# ---------------------------------------------------------------- fp16 tile-heuristic sweep

F16_VARIANTS = [(0, "auto"), (6, "no_pairs"), (5, "whole_tiles"), (9, "k_slices_tail"),
                (10, "stream_k"), (15, "halves_tail"), (14, "stream_k_tail"),
                (12, "width_224"), (13, "width_192")]


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
    clocks = sampler.stop().summary()
    print(json.dumps({"sweep": "fp16 heuristic 1024..12800 step 128", "sizes": len(sizes),
                      "auto_best": best_is_auto, "auto_within_2pct": within, "clocks": clocks}))


# (forced path, k-blocks per ring stage (0 = automatic), name)
TALL_VARIANTS = [(0, 0, "auto"), (5, 1, "whole_tiles"), (5, 2, "whole_tiles_2kb"),
                 (11, 1, "stream_k"), (11, 2, "stream_k_2kb"), (17, 0, "rows_64")]


def run_sweep_tall(args):
    """Tall half-precision GEMMs (C = 0.75*A*B - 0.25*C, N = 64 and 32, so
    64-wide tiles with no half-width units): the automatic choice beside
    whole 128-row tiles in one wave and stream-K over every tile (each with
    one and with two k-blocks per ring stage) and 64-row tiles, each timed
    the same way (L2 cleared before every replay, second-half mean of 24
    replays)."""
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
    ms_list, ks_list = (512, 1024, 2048, 4096, 6144, 8192, 9728), (512, 1024, 2048, 4096, 8192, 16384)
    max_mk = 9728 * 16384
    seed = synthetic.config_seed(6)
    A, _ = _fill_device((max_mk,), np.float16, seed, synthetic.STREAM_A)
    B, _ = _fill_device((16384 * 64,), np.float16, seed, synthetic.STREAM_B)
    C, _ = _fill_device((9728 * 64,), np.float16, seed, synthetic.STREAM_C)
    sampler = ClockSampler(0).start()
    n = auto_best = within_1us = 0
    lost_us = 0.0
    for N in (64, 32):
        for M in ms_list:
            for K in ks_list:
                if M * K > max_mk:
                    continue
                rec = {"M": M, "N": N, "K": K}
                for path, kpb, name in TALL_VARIANTS:
                    prev = g.force_path(path)
                    prev_k = g.stage_kblocks(kpb)
                    try:
                        fn = lambda: g.gemm_f16(A, B, C, 0.75, -0.25, M=M, N=N, K=K, lda=K, ldb=N,
                                                ldc=N, stream=stream)
                        ms = timed_replays(fn, 24, 3, stream, flush)
                        rec[name] = {"us": round(second_half_mean(ms) * 1e3, 2),
                                     "path": g.last_path()}
                    finally:
                        g.force_path(prev)
                        g.stage_kblocks(prev_k)
                best = min(v["us"] for v in rec.values() if isinstance(v, dict))
                rec["auto_minus_best_us"] = round(rec["auto"]["us"] - best, 2)
                n += 1
                auto_best += rec["auto"]["us"] <= best
                within_1us += rec["auto_minus_best_us"] <= 1.0
                lost_us += rec["auto_minus_best_us"]
                if out:
                    out.write(json.dumps(rec) + "\n")
                    out.flush()
    clocks = sampler.stop().summary()
    print(json.dumps({"sweep": "fp16 tall M 512..9728 x N 32, 64 x K 512..16384", "shapes": n,
                      "auto_best": auto_best, "auto_within_1us": within_1us,
                      "auto_lost_us_total": round(lost_us, 1), "clocks": clocks}))


# ---------------------------------------------------------------- profiler cases

def run_ncu_case(case):
    """One workload of the line, five calls with the L2 flushed before each and
    nothing else: the program a profiler capture of one kernel attaches to."""
    import torch
    import dense_gemm_03_gb300 as g
    import synthetic
    from dense_gemm_03_gb300 import build as _b
    _b.build()
    torch.cuda.set_device(0)
    if case in ("f16", "f32", "ffma"):
        dt = np.float16 if case == "f16" else np.float32
        seed = synthetic.config_seed(2 if case == "f16" else 1)
        A, _ = _fill_device((4096, 4096), dt, seed, synthetic.STREAM_A)
        B, _ = _fill_device((4096, 4096), dt, seed, synthetic.STREAM_B)
        C, _ = _fill_device((4096, 4096), dt, seed, synthetic.STREAM_C)
        if case == "f16":
            fn = lambda: g.gemm_f16(A, B, C, F16_CFG["alpha"], F16_CFG["beta"])
        else:
            fn = lambda: g.sgemm_f32(A, B, C, 1.0, 0.0)
        if case == "ffma":
            g.force_path(PATH_FFMA_ONLY)
    else:
        sM, sN, sK, slda, alpha, beta, _ = EDGE_SHAPES[["edge", "skinny", "tall"].index(case)]
        seed = synthetic.config_seed(4)
        A, _ = _fill_device((sM * slda,), np.float16, seed, synthetic.STREAM_A)
        B, _ = _fill_device((sK, sN), np.float16, seed, synthetic.STREAM_B)
        C, _ = _fill_device((sM, sN), np.float16, seed, synthetic.STREAM_C)
        fn = lambda: g.gemm_f16(A, B, C, alpha, beta, M=sM, N=sN, K=sK, lda=slda, ldb=sN, ldc=sN)
    for _ in range(5):
        g.l2_flush(0)
        fn()
    torch.cuda.synchronize()
    assert g.debug_status() == 0
    print(json.dumps({"ncu_case": case, "kernel_path": g.last_path()}))


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
    ap.add_argument("--sustain-seconds", type=float, default=2.0,
                    help="headline replays back to back afterwards (clock samples under load)")
    ap.add_argument("--no-tf32-peak", action="store_true",
                    help="skip measuring the dense tf32 rate (3xTF32 denominator)")
    ap.add_argument("--f32-ffma", action="store_true",
                    help="time the fp32 leg on the CUDA-core FFMA kernel instead of 3xTF32")
    ap.add_argument("--ncu-case", choices=["f16", "f32", "ffma", "skinny", "tall", "edge"],
                    default=None,
                    help="run one workload five times (L2 flushed before each) and exit: the "
                         "small case a profiler capture attaches to")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-f16", action="store_true",
                    help="fp16 sweep: the automatic path beside the forced alternatives")
    ap.add_argument("--sweep-tall", action="store_true",
                    help="fp16 tall shapes: the automatic schedule beside the forced ones")
    ap.add_argument("--sweep-out", default=None)
    ap.add_argument("--sweep-sizes", default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return
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
    if args.sweep_tall:
        run_sweep_tall(args)
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
