#!/usr/bin/env python3
"""Benchmark of libhgemm on the GEMM workloads; prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload square4096|square8192|batched_qk|ragged4095|
                                ragged4095_h|skinny|int512]

A step is one product C = A.B of the workload (every step of the hot path:
operand copies when an operand is misaligned, the tensor-core kernel and its
epilogue), with inputs already resident in HBM.  The default workload is the
4096^3 bf16 GEMM (N(0,1) inputs, seed 1, bf16 out), the configuration the
metric is quoted on.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and ``torch.cuda.synchronize()``; CUDA events on the launching stream time the
whole region and every launch.  L2 is defeated by rotating enough copies of
the inputs and outputs that the working set exceeds twice the L2 size.
Clocks and throttle reasons are sampled with nvidia-smi while the GPU is under
load (the timed region, extended by an untimed probe loop when the region is
shorter than the sampling period).

Multi-GPU: the product does not shard in this library (every box runs one
GPU), so ``--gpus N`` under torchrun runs N independent replicas; ``value`` is
the FLOPs of all ranks divided by the slowest rank's time.

``--impl reference`` times the CPU oracle (the only other implementation of
the method) on the host cores on a bounded sample of the same workload.

The default run (square4096) also measures every other GEMM configuration
the method is judged on -- int512, square8192, batched_qk, ragged4095,
ragged4095_h and skinny -- one after the other, outside the headline's timed
region, and adds them to the same JSON line as ``per_config``: each with its
own timed region (about half a second of back-to-back launches, L2 defeated
the same way), roofline fraction, percentage of the stated peaks, the
stated target when there is one, and clocks.  Each entry's ``cpu_baseline``
times the oracle on sampled entries of that configuration's C and reports,
from the same sample, the GPU result's normalised error
(``max |C - Cref| / sum_k |A_ik||B_kj|``; int512 is compared in full, bit for
bit).  ``--no-per-config`` skips them.
"""
from __future__ import annotations

import argparse
import glob
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s at 1 GB300 and % of dense fp16/bf16 tensor peak (or % HBM BW)"
NOMINAL_TC_TFLOPS = 2250.0   # dense fp16/bf16 per GPU, nominal
NOMINAL_F8_RATIO = 2.0       # dense fp8 / dense bf16 tensor rate, nominal (4.5 / 2.25 PFLOP/s)
F8_TYPES = ("e4m3", "e5m2")
ORACLE_IN = {"f16": 0, "bf16": 1, "e4m3": 2, "e5m2": 3}  # the oracle's input-type codes
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 2**20
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="square4096")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other configurations (default run only)")
    ap.add_argument("--per-config-seconds", type=float, default=0.5,
                    help="length of each configuration's timed region")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--epilogue", choices=["none", "bias_gelu", "bias_gelu_tanh", "beta_bias_relu"],
                    default="none",
                    help="fused epilogue on every step (hgemm_run_ex): bias + GELU (erf or tanh "
                         "form), or beta = 1 (reads C) + bias + ReLU")
    ap.add_argument("--probe-seconds", type=float, default=1.0,
                    help="untimed load after the timed region so the clock sampler sees the GPU busy")
    ap.add_argument("--shape", default=None,
                    help="M,N,K: the workload's inputs (types, distributions, seed) at another "
                         "size, for profiling captures; implies --no-per-config")
    ap.add_argument("--plan-options", default="",
                    help="comma-separated hgemm_options_t fields for the timed plans, e.g. "
                         "cta_pair=2,force_generic_store=1 (recorded in config)")
    return ap.parse_args()


def plan_options(args, w):
    """hgemm_options_t of the timed plans: the workload's B layout plus
    --plan-options."""
    from tensor_core_dense_swizzled_gb300 import hgemm as H
    kw = {"trans_b": int(w.trans_b)}
    for item in filter(None, (x.strip() for x in args.plan_options.split(","))):
        k, _, v = item.partition("=")
        if k not in dict(H.Options._fields_):
            raise SystemExit(f"--plan-options: unknown field {k}")
        kw[k] = int(v)
    return H.Options(**kw)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16": d["bf16_tflops"], "bf16_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "hbm": d["hbm_gbs"], "source": "measured"}
    except Exception:
        return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def whole_job_tflops(flops_per_step: int, steps: int, world: int, slowest_region_ms: float) -> float:
    """Replicas: every rank runs `steps` products; the job's throughput is all
    ranks' FLOPs over the slowest rank's timed region."""
    return flops_per_step * steps * world / (slowest_region_ms * 1e-3) / 1e12


def max_over_ranks(pg, x: float, device) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        sm, smax, reasons = [], [], set()
        for ts, line in self.lines:
            if ts < t0 or ts > t1:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- helpers

def kernel_family(kernel_name: str) -> str:
    for fam in ("pair", "tiled", "skinny"):
        if f"hgemm_{fam}_kernel" in kernel_name:
            return fam
    return "attention" if "attention" in kernel_name else "other"


# Headers every kernel is compiled with (the host-only ones, hgemm.h and
# internal.h, do not reach device code and are left out).
DEVICE_HEADERS = ("kernels.h", "ptx.cuh", "tile_common.cuh", "watchdog.cuh")


def kernel_hash(family: str, csrc: str | None = None) -> str:
    """Hash of the device sources a kernel family is built from: its own
    files and the headers device code includes (the stored entry names the
    kernel variant the capture saw)."""
    own = {
        "pair": ("gemm_pair",),
        "tiled": ("gemm_tiled",),
        "skinny": ("gemm_skinny",),
        "attention": ("attention.cu",),
    }.get(family, ())
    csrc = csrc or os.path.join(ROOT, "tensor_core_dense_swizzled_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(csrc, "*"))):
        base = os.path.basename(f)
        if base not in DEVICE_HEADERS and not base.startswith(own):
            continue
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch of the main kernel from a committed ncu capture,
    or None when absent or taken on other sources of that kernel family."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_hash") == kernel_hash(kernel_family(e.get("kernel", ""))):
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def flops_of(w):
    return 2 * w.M * w.N * w.K * w.batch


def in_bytes_of(w) -> int:
    return 1 if w.dtype_in in F8_TYPES else 2


def tensor_ratio(w) -> float:
    """Tensor-core rate of the workload's input type relative to bf16."""
    return NOMINAL_F8_RATIO if w.dtype_in in F8_TYPES else 1.0


def min_bytes_of(w):
    ob = 4 if w.dtype_out == "f32" else 2
    ib = in_bytes_of(w)
    return w.batch * (w.M * w.K * ib + w.K * w.N * ib + w.M * w.N * ob), ob


def roofline_bound(w) -> str:
    fl = flops_of(w)
    by, _ = min_bytes_of(w)
    ridge = NOMINAL_TC_TFLOPS * tensor_ratio(w) * 1e12 / (NOMINAL_HBM_GBS * 1e9)
    return "tensor" if fl / by > ridge else "hbm"


# ---------------------------------------------------------------- CPU oracle

def oracle_rows_time(w, A_bits, B_bits, rows: int, threads: int) -> float:
    import oracle
    din = ORACLE_IN[w.dtype_in]
    t0 = time.perf_counter()
    if w.trans_b:  # the transposition is part of the oracle's work
        oracle.gemm_bt(A_bits[: max(1, rows * w.lda)], B_bits[: w.N * w.ldb], din, rows, w.N, w.K,
                       w.lda, w.ldb, 1, 0, 0)
    else:
        oracle.gemm(A_bits[: max(1, rows * w.lda)],
                    B_bits[: (w.K - 1) * w.ldb + w.N] if w.batch == 1 else B_bits,
                    din, rows, w.N, w.K, w.lda, w.ldb, 1, 0, 0, threads=threads)
    return time.perf_counter() - t0


def cpu_inputs(w):
    import numpy as np
    import torch

    from tensor_core_dense_swizzled_gb300 import inputs
    A, B = inputs.make_inputs(w)
    if w.dtype_in in F8_TYPES:  # 8-bit patterns widened to the oracle's 16-bit arrays
        ab = A.contiguous().view(torch.uint8).numpy().astype(np.uint16).reshape(-1)
        bb = B.contiguous().view(torch.uint8).numpy().astype(np.uint16).reshape(-1)
        return ab, bb
    ab = A.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    bb = B.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return ab, bb


def cpu_baseline(w, target_s: float = 12.0):
    """Times the oracle, as it stands, on the host cores on whole rows of C of
    batch 0 (a bounded sample of the workload); returns the cpu_baseline dict."""
    ab, bb = cpu_inputs(w)
    threads = os.cpu_count() or 1
    rows = min(w.M, threads)
    t = oracle_rows_time(w, ab, bb, rows, threads)
    per_row = t / rows
    rows = int(max(threads, min(w.M, math.floor(target_s / max(per_row, 1e-9) / threads) * threads)))
    rows = min(rows, w.M)
    t = oracle_rows_time(w, ab, bb, rows, threads)
    fl = 2 * rows * w.N * w.K
    return {"value": fl / t / 1e12, "unit": "TFLOP/s", "cores": min(threads, rows), "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of C (batch 0) of {w.name}: {rows}x{w.N}x{w.K}, "
                      f"fp64 triple loop, {t:.1f} s"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return 0
    ab, bb = cpu_inputs(w)
    threads = os.cpu_count() or 1
    # size each step so that warm-up + timed steps take about 90 s in total
    t1 = oracle_rows_time(w, ab, bb, min(w.M, threads), threads) / min(w.M, threads) * threads
    per_step_budget = 90.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(w.M, math.floor(per_step_budget / max(t1 / threads, 1e-9)))))
    for _ in range(args.warmup):
        oracle_rows_time(w, ab, bb, rows, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_rows_time(w, ab, bb, rows, threads)
    dt = time.perf_counter() - t0
    fl = 2 * rows * w.N * w.K * args.steps
    value = fl / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": min(threads, rows), "kind": "oracle",
                         "sample": f"each step: rows 0..{rows - 1} of C of {w.name} ({rows}x{w.N}x{w.K})"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# The targets stated for the configurations: a fraction of the stated dense
# fp16/bf16 tensor peak (2.25 PFLOP/s) or of the stated HBM bandwidth (8 TB/s).
STATED_TARGETS = {"square4096": ("tensor", 0.70), "square8192": ("tensor", 0.70),
                  "skinny": ("hbm", 0.70)}
PER_CONFIG = ("int512", "square8192", "batched_qk", "ragged4095", "ragged4095_h", "skinny")
# acceptance bound on max |C - Cref| / Den per output type (bf16: the provable
# 5e-3; the stated 4e-3 for 16-bit output is reported beside it)
PARITY_TOL = {"f32": 1e-3, "f16": 4e-3, "bf16": 5e-3}
STATED_16BIT_TOL = 4e-3


def kernel_label(info) -> str:
    """Which kernel a plan runs: pair (256 x 256 tiles on CTA pairs), single
    (one CTA per 128 x tile_n tile) or skinny; "+copy" when an operand is
    first copied to an aligned buffer."""
    if info["path"] == 3:
        k = "skinny"
    elif info["path"] == 2:
        k = "pair" if info["tile_m"] == 256 else "single"
    else:
        return {0: "empty", 1: "zero_fill"}.get(info["path"], "?")
    return k + ("+copy" if info["repack_a"] or info["repack_b"] else "")


def stated_target(w, tflops: float, gbs: float):
    t = STATED_TARGETS.get(w.name)
    if t is None:
        return None
    kind, frac = t
    if kind == "tensor":
        got = tflops / (NOMINAL_TC_TFLOPS * tensor_ratio(w))
        return {"target": f">= {frac:.0%} of the stated {NOMINAL_TC_TFLOPS:g} TFLOP/s dense tensor peak",
                "fraction": got, "met": got >= frac}
    got = gbs / NOMINAL_HBM_GBS
    return {"target": f">= {frac:.0%} of the stated {NOMINAL_HBM_GBS:g} GB/s HBM bandwidth",
            "fraction": got, "met": got >= frac}


def config_of(w, world, extra=None):
    c = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "batch": w.batch, "dtype_in": w.dtype_in,
         "dtype_out": w.dtype_out, "seed": w.seed, "parallelism": "replicas" if world > 1 else "single",
         "layout": ("A MxK, B NxK (C = A.B^T)" if w.trans_b else "A MxK, B KxN") + ", C MxN row-major"}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------- per-configuration runs

def config_cpu_check(w, A, B, C_dev, sample_entries: int = 1024, seed: int = 99):
    """The cpu_baseline leg of one configuration: times the oracle, as it
    stands, on a sample of C's entries (every entry for int512, whose product
    the oracle computes in a fraction of a second), and compares the GPU's C
    with it there.  Returns (cpu_baseline, parity)."""
    import numpy as np
    import torch

    import oracle
    ab = A.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    bb = B.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
    din = ORACLE_IN[w.dtype_in]
    C = C_dev.reshape(w.batch, w.M, w.N)
    threads = os.cpu_count() or 1
    if w.name == "int512":
        t0 = time.perf_counter()
        Cref, Den = oracle.gemm(ab, bb, din, w.M, w.N, w.K, w.lda, w.ldb, w.batch, w.strideA,
                                w.strideB, threads=threads)
        dt = time.perf_counter() - t0
        got = C.double().cpu().numpy()
        exact = bool(np.array_equal(got, Cref))
        cpu = {"value": flops_of(w) / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"the whole {w.M}x{w.N}x{w.K} product, {dt:.2f} s"}
        return cpu, {"entries": w.M * w.N, "bit_exact": exact,
                     "max_normalised_error": oracle.normalized_error(got, Cref, Den), "pass": exact}
    rng = np.random.default_rng(seed)
    eb = rng.integers(0, w.batch, sample_entries)
    ei = rng.integers(0, w.M, sample_entries)
    ej = rng.integers(0, w.N, sample_entries)
    # the corners and the last row and column (ragged edges)
    eb = np.concatenate([eb, [0, 0, w.batch - 1, w.batch - 1], np.full(32, w.batch - 1),
                         np.full(32, w.batch - 1)])
    ei = np.concatenate([ei, [0, w.M - 1, 0, w.M - 1], np.full(32, w.M - 1), rng.integers(0, w.M, 32)])
    ej = np.concatenate([ej, [0, w.N - 1, w.N - 1, 0], rng.integers(0, w.N, 32), np.full(32, w.N - 1)])
    vals = C[torch.as_tensor(eb, device=C.device), torch.as_tensor(ei, device=C.device),
             torch.as_tensor(ej, device=C.device)].cpu()
    if w.dtype_out == "f32":
        got = vals.double().numpy()
    else:
        got = oracle.decode(vals.view(torch.int16).numpy().view(np.uint16), ORACLE_IN[w.dtype_out])
    t0 = time.perf_counter()
    cref, den = oracle.gemm_entries(ab, bb, din, w.K, w.lda, w.ldb, eb, ei, ej, w.strideA, w.strideB)
    dt = time.perf_counter() - t0
    err = oracle.normalized_error(got, cref, den)
    cpu = {"value": 2 * eb.size * w.K / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
           "sample": f"{eb.size} entries of C (random, corners, last row and column), "
                     f"one fp64 dot product of length {w.K} each, {dt * 1e3:.0f} ms"}
    par = {"entries": int(eb.size), "max_normalised_error": err, "tolerance": PARITY_TOL[w.dtype_out],
           "pass": err <= PARITY_TOL[w.dtype_out]}
    if w.dtype_out != "f32":
        par["stated_tolerance"] = STATED_16BIT_TOL
        par["pass_stated"] = err <= STATED_16BIT_TOL
    return cpu, par


def measure_config(name, H, dev, stream, sampler, peaks, seconds: float, with_cpu: bool):
    """One configuration in the launch configuration of the headline: rotating
    input/output sets larger than 2 x L2, warm-up, then back-to-back launches
    for about `seconds` between two CUDA events on the launching stream."""
    import torch

    from tensor_core_dense_swizzled_gb300 import inputs
    DT = {"f16": H.HGEMM_F16, "bf16": H.HGEMM_BF16, "f32": H.HGEMM_F32}
    TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    w = inputs.WORKLOADS[name]
    A, B = inputs.make_inputs(w)
    fl = flops_of(w)
    min_bytes, ob = min_bytes_of(w)
    set_bytes = (A.numel() + B.numel()) * in_bytes_of(w) + w.batch * w.M * w.N * ob
    nsets = max(1, math.ceil(2 * L2_BYTES / set_bytes))
    shape_c = (w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N)
    sets, plans = [], []
    try:
        for _ in range(nsets):
            sets.append((A.to(dev), B.to(dev), torch.empty(shape_c, dtype=TD[w.dtype_out], device=dev)))
            plans.append(H.hgemm_plan_create_ex(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, w.batch, w.strideA,
                                                w.strideB, w.strideC, DT[w.dtype_in], DT[w.dtype_out],
                                                H.Options(trans_b=int(w.trans_b))))
        info = H.hgemm_plan_get_info(plans[0])

        def run(n, i0=0):
            for i in range(i0, i0 + n):
                a, b, c = sets[i % nsets]
                H.hgemm_run(plans[i % nsets], a, b, c, stream)

        run(max(5, nsets))
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(20)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        est_ms = e0.elapsed_time(e1) / 20
        steps = int(min(20000, max(100, round(seconds * 1e3 / max(est_ms, 1e-3)))))
        torch.cuda.synchronize(dev)
        t_wall0 = time.time()
        e0.record(stream)
        run(steps)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t_wall1 = time.time()
        region_ms = e0.elapsed_time(e1)
        for p in plans:
            st = H.hgemm_check(p, stream)
            if st != 0:
                raise RuntimeError(f"{name}: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}")
        clocks = sampler.summary(t_wall0, t_wall1)
        ms = region_ms / steps
        tflops = fl / (ms * 1e-3) / 1e12
        gbs = min_bytes / (ms * 1e-3) / 1e9
        bound = roofline_bound(w)
        sustained = region_ms > 1000.0
        if bound == "tensor":
            peak = (peaks["bf16_sustained"] if sustained else peaks["bf16"]) * tensor_ratio(w)
            roof = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                    "frac": tflops / peak,
                    "peak_kind": ("sustained" if sustained else "burst") + f" bf16, {peaks['source']}"}
        else:
            roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm"], "peak_kind": f"copy bandwidth, {peaks['source']}"}
        roof["traffic"] = committed_traffic(w.name)
        roof["kernels_per_launch"] = info["kernels_per_run"]
        entry = {
            "workload": name, "M": w.M, "N": w.N, "K": w.K, "batch": w.batch, "dtype_in": w.dtype_in,
            "dtype_out": w.dtype_out, "seed": w.seed, "kernel": kernel_label(info),
            "tile": [info["tile_m"], info["tile_n"], info["tile_k"]], "grid": info["grid"],
            "steps": steps, "ms_per_step": ms, "value": tflops, "unit": "TFLOP/s", "gbs": gbs,
            "pct_nominal_tensor_peak": 100.0 * tflops / (NOMINAL_TC_TFLOPS * tensor_ratio(w)),
            "pct_nominal_hbm": 100.0 * gbs / NOMINAL_HBM_GBS, "roofline": roof,
            "stated_target": stated_target(w, tflops, gbs), "clocks": clocks,
            "l2": f"{nsets} rotating sets ({nsets * set_bytes / 2**20:.0f} MiB)",
        }
        if with_cpu:
            entry["cpu_baseline"], entry["parity"] = config_cpu_check(w, A, B, sets[0][2])
        return entry, steps * info["kernels_per_run"]
    finally:
        for p in plans:
            H.hgemm_plan_destroy(p)
        del sets
        torch.cuda.empty_cache()


# ---------------------------------------------------------------- GPU arm

def run_ours(args, w, world, rank, local, pg):
    import torch

    import __graft_entry__
    from tensor_core_dense_swizzled_gb300 import hgemm as H
    from tensor_core_dense_swizzled_gb300 import inputs

    __graft_entry__.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    DT = {"f16": H.HGEMM_F16, "bf16": H.HGEMM_BF16, "f32": H.HGEMM_F32, "e4m3": H.HGEMM_E4M3,
          "e5m2": H.HGEMM_E5M2}
    TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    A, B = inputs.make_inputs(w)
    flops = flops_of(w)
    min_bytes, ob = min_bytes_of(w)
    ib = in_bytes_of(w)
    set_bytes = A.numel() * ib + B.numel() * ib + w.batch * w.M * w.N * ob
    nsets = max(1, math.ceil(2 * L2_BYTES / set_bytes))
    shape_c = (w.batch, w.M, w.N) if w.batch > 1 else (w.M, w.N)
    sets, plans = [], []
    for _ in range(nsets):
        sets.append((A.to(dev), B.to(dev), torch.empty(shape_c, dtype=TD[w.dtype_out], device=dev)))
        plans.append(H.hgemm_plan_create_ex(w.M, w.N, w.K, w.lda, w.ldb, w.ldc, w.batch, w.strideA,
                                            w.strideB, w.strideC, DT[w.dtype_in], DT[w.dtype_out],
                                            plan_options(args, w)))
    info = H.hgemm_plan_get_info(plans[0])
    stream = torch.cuda.current_stream(dev)

    epi = None
    if args.epilogue != "none":
        import types
        gen = torch.Generator().manual_seed(w.seed + 99)
        bias_dev = torch.randn(w.N, generator=gen).to(dev)
        epi = types.SimpleNamespace(
            alpha=1.0, beta=1.0 if args.epilogue == "beta_bias_relu" else 0.0, bias=bias_dev,
            row_scale=None, col_scale=None,
            activation={"bias_gelu": H.HGEMM_ACT_GELU, "bias_gelu_tanh": H.HGEMM_ACT_GELU_TANH,
                        "beta_bias_relu": H.HGEMM_ACT_RELU}[args.epilogue])
        for a_, b_, c_ in sets:
            c_.zero_()  # beta = 1 reads C: start from defined values

    def step(i):
        a, b, c = sets[i % nsets]
        if epi is None:
            H.hgemm_run(plans[i % nsets], a, b, c, stream)
        else:
            H.hgemm_run_ex(plans[i % nsets], a, b, c, epi, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    st = H.hgemm_check(plans[0], stream)
    if st != 0:
        raise RuntimeError(f"warm-up failed: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)  # let nvidia-smi come up
    # Events only at the two ends of the timed region: an event between two
    # launches would stop the next one from starting early (dependent
    # launches), which a caller's back-to-back stream does not do.
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ev_start.record(stream)
    for i in range(args.steps):
        step(i)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(pg)
    t_wall1 = time.time()
    region_ms = ev_start.elapsed_time(ev_end)
    # keep the GPU busy (untimed) long enough for the clock sampler to see it
    probe_until = t_wall0 + args.probe_seconds
    j = 0
    while time.time() < probe_until:
        for _ in range(50):
            step(j)
            j += 1
        torch.cuda.synchronize(dev)
    t_wall2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0 - 0.05, max(t_wall1, t_wall2) + 0.05)
    clocks["window"] = "timed" if t_wall1 - t_wall0 >= 1.0 else "timed+probe"
    st = H.hgemm_check(plans[0], stream)
    if st != 0:
        raise RuntimeError(f"timed run failed: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}")

    region_ms = max_over_ranks(pg, region_ms, dev)
    value = whole_job_tflops(flops, args.steps, world, region_ms)
    # one hgemm_run per step: its kernels back to back (one kernel except when
    # an operand copy precedes the GEMM, kernels_per_launch = 2, where this
    # average covers both and the achieved rate is conservative)
    avg_launch_ms = region_ms / args.steps
    bound = roofline_bound(w)
    peaks = load_peaks()
    sustained = region_ms > 1000.0
    if bound == "tensor":
        achieved = flops / (avg_launch_ms * 1e-3) / 1e12
        # an 8-bit contraction: the measured bf16 peak x the nominal fp8 / bf16 ratio
        peak = (peaks["bf16_sustained"] if sustained else peaks["bf16"]) * tensor_ratio(w)
        unit = "TFLOP/s"
        peak_kind = ("sustained" if sustained else "burst") + f" bf16, {peaks['source']}"
        if tensor_ratio(w) != 1.0:
            peak_kind += f", x {tensor_ratio(w):g} (nominal fp8 / bf16 rate)"
    else:
        achieved = min_bytes / (avg_launch_ms * 1e-3) / 1e9
        peak = peaks["hbm"]
        unit = "GB/s"
        peak_kind = f"copy bandwidth, {peaks['source']}"
    roof = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": committed_traffic(w.name), "peak_kind": peak_kind,
            "algorithmic_per_launch": flops if bound == "tensor" else min_bytes,
            "launch_ms": avg_launch_ms, "kernels_per_launch": info["kernels_per_run"]}

    # end to end through the C ABI with host buffers (copies inside the timed region)
    e2e = None
    if args.e2e_steps > 0:
        Ah = A.pin_memory()
        Bh = B.pin_memory()
        Ch = torch.empty(shape_c, dtype=TD[w.dtype_out]).pin_memory()
        H.hgemm_run_host(plans[0], Ah, Bh, Ch, stream)  # allocates the staging buffers
        barrier(pg)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            H.hgemm_run_host(plans[0], Ah, Bh, Ch, stream)
        dt = time.perf_counter() - t0
        dt = max_over_ranks(pg, dt, dev)
        e2e = {"value": flops * args.e2e_steps * world / dt / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": A.numel() * ib + B.numel() * ib,
               "d2h_bytes_per_step": w.batch * w.M * w.N * ob, "steps": args.e2e_steps}
        e2e.update(host_link_rates(Ah, Bh, Ch, sets[0], stream, dev))
        chunks = info.get("host_chunks", 1)
        e2e["copies"] = (f"{chunks} row chunks: copies in, products and copies out overlap on three "
                         "streams" if chunks > 1 else "serialised with the kernel on one stream")
        e2e["ms_per_step"] = dt / args.e2e_steps * 1e3

    for p in plans:
        H.hgemm_plan_destroy(p)
    del sets
    torch.cuda.empty_cache()

    # the other configurations, each with its own timed region (after the
    # headline's, so they do not change it)
    per_config = None
    if (world == 1 and w.name == "square4096" and args.epilogue == "none"
            and not args.no_per_config):
        per_config = []
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.3)
        try:
            for name in PER_CONFIG:
                entry, _ = measure_config(name, H, dev, stream, sampler, load_peaks(),
                                          args.per_config_seconds, not args.no_cpu_baseline)
                per_config.append(entry)
        finally:
            sampler.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": region_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype_in, "data": "synthetic",
        "config": config_of(w, world, {
            "l2": f"{nsets} rotating input/output sets ({nsets * set_bytes / 2**20:.0f} MiB > 2x L2)",
            "path": {2: "tiled", 3: "skinny", 1: "zero_fill", 0: "empty"}[info["path"]],
            "kernel": kernel_label(info),
            "tile": [info["tile_m"], info["tile_n"], info["tile_k"]], "stages": info["stages"],
            "split_k": info["split_k"], "grid": info["grid"], "epilogue": args.epilogue,
            **({"plan_options": args.plan_options} if args.plan_options else {})}),
        "pct_nominal_tensor_peak": 100.0 * value / world / (NOMINAL_TC_TFLOPS * tensor_ratio(w)),
        "pct_nominal_hbm": 100.0 * (min_bytes * args.steps / (region_ms * 1e-3) / 1e9) / NOMINAL_HBM_GBS,
        "stated_target": stated_target(w, value / world,
                                       min_bytes * args.steps / (region_ms * 1e-3) / 1e9),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * info["kernels_per_run"],
        "clocks": clocks,
    }
    if per_config is not None:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)
    return 0


def host_link_rates(Ah, Bh, Ch, dev_set, stream, dev, reps: int = 5):
    """Achieved host <-> device copy rates of the step's own buffers (pinned
    host memory), each direction alone: best of `reps`, CUDA events on the
    stream.  They bound the end-to-end step, whose copies and kernel run one
    after the other on one stream."""
    import torch
    dA, dB, dC = dev_set
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    h2d, d2h = [], []
    nb_in = Ah.numel() * Ah.element_size() + Bh.numel() * Bh.element_size()
    nb_out = Ch.numel() * Ch.element_size()
    with torch.cuda.stream(stream):
        for _ in range(reps):
            e0.record(stream)
            dA.copy_(Ah, non_blocking=True)
            dB.copy_(Bh, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            h2d.append(e0.elapsed_time(e1))
            e0.record(stream)
            Ch.copy_(dC, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            d2h.append(e0.elapsed_time(e1))
    return {"h2d_gbs": nb_in / (min(h2d) * 1e-3) / 1e9, "d2h_gbs": nb_out / (min(d2h) * 1e-3) / 1e9}


# ---------------------------------------------------------------- attention

def attn_flops(w) -> int:
    """2 * bh * sq * skv * d for each of S = Q K^T and O = P V; under the
    causal mask only the allowed (query, key) pairs count."""
    if w.causal:
        pairs = sum(min(w.skv, i + 1 + w.skv - w.sq) for i in range(w.sq))
    else:
        pairs = w.sq * w.skv
    return 4 * w.bh * pairs * 128


def attn_config(w, world, extra=None):
    c = {"workload": w.name, "batch_heads": w.bh, "seq_q": w.sq, "seq_kv": w.skv, "head_dim": 128,
         "dtype_in": w.dtype, "dtype_out": w.dtype, "causal": w.causal, "scale": w.scale,
         "seed": w.seed, "parallelism": "replicas" if world > 1 else "single",
         "layout": "Q, K, V, O [bh][seq][128] row-major"}
    if extra:
        c.update(extra)
    return c


def attn_oracle_time(w, qb, kb, vb, rows: int, threads: int) -> float:
    """Oracle attention on query rows 0 .. rows-1 of head 0 (the longest rows
    of a causal head are the last ones: rows are taken from the end then)."""
    import numpy as np

    import oracle
    ri = np.arange(w.sq - rows, w.sq) if w.causal else np.arange(rows)
    rb = np.zeros(rows, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.attention(qb, kb, vb, ORACLE_IN[w.dtype], w.bh, w.sq, w.skv, 128, w.scale, w.causal,
                     rows=(rb, ri), threads=threads)
    return time.perf_counter() - t0


def attn_cpu_inputs(w):
    import numpy as np
    import torch

    from tensor_core_dense_swizzled_gb300 import inputs
    Q, K, V = inputs.make_attention_inputs(w)
    conv = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)  # noqa: E731
    return conv(Q), conv(K), conv(V)


def attn_pairs_of_rows(w, rows: int) -> int:
    if not w.causal:
        return rows * w.skv
    return sum(min(w.skv, i + 1 + w.skv - w.sq) for i in range(w.sq - rows, w.sq))


def attn_cpu_baseline(w, target_s: float = 12.0):
    qb, kb, vb = attn_cpu_inputs(w)
    threads = os.cpu_count() or 1
    rows = min(w.sq, 4 * threads)
    t = attn_oracle_time(w, qb, kb, vb, rows, threads)
    rows = int(min(w.sq, max(threads, math.floor(target_s / max(t / rows, 1e-9) / threads) * threads)))
    t = attn_oracle_time(w, qb, kb, vb, rows, threads)
    fl = 4 * attn_pairs_of_rows(w, rows) * 128
    return {"value": fl / t / 1e12, "unit": "TFLOP/s", "cores": min(threads, rows), "kind": "oracle",
            "sample": f"{rows} query rows of head 0 of {w.name} ({rows} x {w.skv} keys x 128), "
                      f"fp64 loops, {t:.1f} s"}


def run_attention_reference(args, w, rank, world):
    if rank != 0:
        return 0
    qb, kb, vb = attn_cpu_inputs(w)
    threads = os.cpu_count() or 1
    t1 = attn_oracle_time(w, qb, kb, vb, min(w.sq, threads), threads) / min(w.sq, threads)
    per_step_budget = 90.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(w.sq, math.floor(per_step_budget / max(t1, 1e-9)))))
    for _ in range(args.warmup):
        attn_oracle_time(w, qb, kb, vb, rows, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        attn_oracle_time(w, qb, kb, vb, rows, threads)
    dt = time.perf_counter() - t0
    value = 4 * attn_pairs_of_rows(w, rows) * 128 * args.steps / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": attn_config(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": min(threads, rows), "kind": "oracle",
                         "sample": f"each step: {rows} query rows of head 0 of {w.name}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_attention_ours(args, w, world, rank, local, pg):
    import torch

    import __graft_entry__
    from tensor_core_dense_swizzled_gb300 import hgemm as H
    from tensor_core_dense_swizzled_gb300 import inputs

    __graft_entry__.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    DT = {"f16": H.HGEMM_F16, "bf16": H.HGEMM_BF16}
    Q, K, V = inputs.make_attention_inputs(w)
    flops = attn_flops(w)
    set_bytes = (Q.numel() + K.numel() + V.numel() + Q.numel()) * 2
    nsets = max(1, math.ceil(2 * L2_BYTES / set_bytes))
    sets = [(Q.to(dev), K.to(dev), V.to(dev), torch.empty_like(Q, device=dev)) for _ in range(nsets)]
    plan = H.hgemm_attention_plan_create(w.bh, w.sq, w.skv, 128, w.scale, int(w.causal), DT[w.dtype])
    stream = torch.cuda.current_stream(dev)

    def step(i):
        q, k, v, o = sets[i % nsets]
        H.hgemm_attention_run(plan, q, k, v, o, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    st = H.hgemm_attention_check(plan, stream)
    if st != 0:
        raise RuntimeError(f"warm-up failed: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ev_start.record(stream)
    for i in range(args.steps):
        step(i)
    ev_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(pg)
    t_wall1 = time.time()
    region_ms = ev_start.elapsed_time(ev_end)
    probe_until = t_wall0 + args.probe_seconds
    j = 0
    while time.time() < probe_until:
        for _ in range(50):
            step(j)
            j += 1
        torch.cuda.synchronize(dev)
    t_wall2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0 - 0.05, max(t_wall1, t_wall2) + 0.05)
    clocks["window"] = "timed" if t_wall1 - t_wall0 >= 1.0 else "timed+probe"
    st = H.hgemm_attention_check(plan, stream)
    if st != 0:
        raise RuntimeError(f"timed run failed: {H.STATUS.get(st)} {H.hgemm_last_error_detail()}")
    region_ms = max_over_ranks(pg, region_ms, dev)
    value = whole_job_tflops(flops, args.steps, world, region_ms)
    avg_launch_ms = region_ms / args.steps
    peaks = load_peaks()
    sustained = region_ms > 1000.0
    achieved = flops / (avg_launch_ms * 1e-3) / 1e12
    peak = peaks["bf16_sustained"] if sustained else peaks["bf16"]
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": committed_traffic(w.name),
            "peak_kind": ("sustained" if sustained else "burst") + f" bf16, {peaks['source']}",
            "algorithmic_per_launch": flops, "launch_ms": avg_launch_ms, "kernels_per_launch": 1}
    e2e = None
    if args.e2e_steps > 0:
        Qh, Kh, Vh = Q.pin_memory(), K.pin_memory(), V.pin_memory()
        Oh = torch.empty_like(Q).pin_memory()
        H.hgemm_attention_run_host(plan, Qh, Kh, Vh, Oh, stream)
        barrier(pg)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            H.hgemm_attention_run_host(plan, Qh, Kh, Vh, Oh, stream)
        dt = time.perf_counter() - t0
        dt = max_over_ranks(pg, dt, dev)
        e2e = {"value": flops * args.e2e_steps * world / dt / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": (Q.numel() + K.numel() + V.numel()) * 2,
               "d2h_bytes_per_step": Q.numel() * 2, "steps": args.e2e_steps,
               "ms_per_step": dt / args.e2e_steps * 1e3,
               "copies": "serialised with the kernel on one stream"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = attn_cpu_baseline(w)
    H.hgemm_attention_plan_destroy(plan)
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": region_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": attn_config(w, world, {
            "l2": f"{nsets} rotating input/output sets ({nsets * set_bytes / 2**20:.0f} MiB > 2x L2)",
            "path": "attention", "tile": [128, 128, 128], "grid": w.bh * ((w.sq + 127) // 128)}),
        "pct_nominal_tensor_peak": 100.0 * value / world / NOMINAL_TC_TFLOPS,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    from tensor_core_dense_swizzled_gb300 import inputs
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.workload in inputs.ATTENTION_WORKLOADS:
        w = inputs.ATTENTION_WORKLOADS[args.workload]
        world, rank, local, pg = dist_setup(args)
        try:
            if args.impl == "reference":
                return run_attention_reference(args, w, rank, world)
            return run_attention_ours(args, w, world, rank, local, pg)
        finally:
            if pg is not None:
                pg.destroy_process_group()
    if args.workload not in inputs.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from "
                         f"{sorted(inputs.WORKLOADS) + sorted(inputs.ATTENTION_WORKLOADS)}")
    w = inputs.WORKLOADS[args.workload]
    if args.shape:
        import dataclasses
        M, N, K = (int(x) for x in args.shape.split(","))
        w = dataclasses.replace(w, name=f"{w.name}@{M}x{N}x{K}", M=M, N=N, K=K)
        args.no_per_config = True
    world, rank, local, pg = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, w, rank, world)
        return run_ours(args, w, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
