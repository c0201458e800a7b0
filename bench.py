#!/usr/bin/env python3
"""Benchmark of the dense fp16 GEMM D = A·Bᵀ (fp16 in, fp32 accumulate, fp16 out).

One step = one D = A·Bᵀ over the headline workload (M = N = K = 8192,
entries normal(0, 1/√K), seeded) through the C ABI, with the operands
already resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

--impl reference times the CPU oracle instead (the only other code that
computes the same D), on this machine's host cores, on a bounded sample of
the same workload (a block of output rows per step).

Under torchrun with N > 1 ranks every rank runs its own replica of the
workload on its own GPU (the GEMM has no exchange step); the value is the
work of all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dense_fp16_gemm_f16_gb300 import inputs, metrics  # noqa: E402

METRIC = "fp16 GEMM TFLOPS (2MNK/t) at 8192³ on 1 GB300; % of dense-fp16 tensor peak"
FP8 = ("e4m3", "e5m2")


def metric_of(dtype: str) -> str:
    """The metric line for an operand type (the fp16 one is the headline)."""
    if dtype in FP8:
        return f"{dtype} GEMM TFLOPS (2MNK/t), bf16 out, on 1 GB300; % of dense-fp8 tensor peak"
    return METRIC
UNIT = "TFLOP/s"
FALLBACK_PEAK_TFLOPS = 1900.0      # used only if the measured-peaks file is absent
L2_ROTATE_BYTES = 256 << 20        # about twice the 129 MB L2
CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=inputs.HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--shape", type=int, nargs=3, metavar=("M", "N", "K"),
                    help="time an M x N x K problem (normal(0, 1/sqrt(K)) entries) instead of a named workload")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--dtype", choices=["f16", "bf16", "e4m3", "e5m2"], default="f16",
                    help="operand type: bf16 runs the same kernels with bf16 operands and output; the 8-bit "
                         "types run the kind::f8f6f4 kernels on amax-scaled operands (one scale for A, one "
                         "per row of B, applied in the fused epilogue) with a bf16 output")
    ap.add_argument("--epilogue", action="store_true",
                    help="time D = relu(1.5 * A·Bᵀ + 0.5 * C + bias) through gemm_nt_ex instead of the plain product")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload record of the other named fp16 workloads")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


# ---------------------------------------------------------------- host-side helpers
def max_over_ranks(pg, x: float, device) -> float:
    """The largest x over all ranks (the slowest rank's time); x itself with one rank."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, M: int, N: int, K: int, ms_max: float) -> float:
    """Whole-job throughput: every rank ran one M x N x K product per step (replicas),
    timed by the slowest rank."""
    return world * metrics.tflops(M, N, K, ms_max * 1e-3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


_COMMENT = re.compile(r"/\*.*?\*/|//[^\n]*", re.S)


def code_of(text: str) -> str:
    """C/CUDA source with comments dropped and white space collapsed (the sources
    hold no string literal with a comment marker)."""
    return " ".join(_COMMENT.sub(" ", text).split())


def source_digest() -> str:
    """sha256 over the code of the CUDA sources (comments and layout ignored):
    identifies the kernel the ncu counters were taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp16_gemm_f16_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode())
                h.update(code_of(f.read()).encode())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("source_sha256") != source_digest():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the benchmark runs."""

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.samples = []
        self.window = None
        self._stop = threading.Event()
        self._proc = None
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
               "-i", str(gpu_index), "-lms", str(period_ms)]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self._proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self._proc is None:
            return None
        time.sleep(0.15)
        self._proc.terminate()
        try:
            self._proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self._proc.kill()
        self._thread.join(timeout=5)
        rows = self.samples
        if self.window:
            inside = [s for s in rows if self.window[0] <= s[0] <= self.window[1]]
            rows = inside if inside else rows
        if not rows:
            return None

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[0]) for _, p in rows if num(p[0]) is not None]
        smax = [num(p[1]) for _, p in rows if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in rows for i in range(4) if p[4 + i].lower() == "active"})
        power = [num(p[2]) for _, p in rows if num(p[2]) is not None]
        mem = [num(p[8]) for _, p in rows if len(p) > 8 and num(p[8]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "mem_mhz": statistics.median(mem) if mem else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


def device_info(gpu_index: int) -> dict:
    """GPU name, driver and CUDA versions of the box the line was measured on."""
    import torch
    info = {"gpu": torch.cuda.get_device_name(gpu_index), "cuda_runtime": torch.version.cuda,
            "torch": torch.__version__}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version,clocks.max.mem", "--format=csv,noheader,nounits",
                              "-i", str(gpu_index)], capture_output=True, text=True, timeout=20).stdout.strip()
        parts = [p.strip() for p in out.split(",")]
        if len(parts) >= 2:
            info["driver"] = parts[0]
            info["mem_max_mhz"] = float(parts[1]) if parts[1].replace(".", "", 1).isdigit() else parts[1]
    except (OSError, subprocess.TimeoutExpired):
        pass
    return info


# ---------------------------------------------------------------- CPU oracle leg
def oracle_rows_fn(A, B, dtype="f16", epi=None, scales=(None, None)):
    """f(r0, r1, threads): the oracle's rows r0..r1-1 of D for this bench configuration."""
    import oracle
    o = oracle.default()
    if dtype == "f16" and epi is None:
        return lambda r0, r1, threads: o.gemm_rows(A, B, r0, r1, nthreads=threads)
    C, bias = epi if epi is not None else (None, None)
    alpha, beta, relu = (EPI_ALPHA, EPI_BETA, True) if epi is not None else (1.0, 0.0, False)
    a_scale, b_scale = scales
    if a_scale is not None:
        alpha = float(np.float32(alpha * a_scale))     # the fp32 alpha the GPU receives
    return lambda r0, r1, threads: oracle._gemm_ex(o, A, B, dtype, alpha, beta, C, bias, relu,
                                                   row_begin=r0, row_end=r1, nthreads=threads,
                                                   scale_n=b_scale)


def oracle_rows_timing(A, B, target_s: float, max_rows: int | None = None, dtype="f16", epi=None,
                       scales=(None, None)):
    """Time the oracle on a block of output rows sized to take about target_s."""
    import oracle
    threads = oracle.default_threads()
    fn = oracle_rows_fn(A, B, dtype, epi, scales)
    M, K = A.shape
    t = time.perf_counter()
    fn(0, 1, threads)
    one = max(time.perf_counter() - t, 1e-4)
    rows = int(max(1, min(M, target_s / one)))
    if max_rows:
        rows = min(rows, max_rows)
    t = time.perf_counter()
    fn(0, rows, threads)
    dt = time.perf_counter() - t
    return rows, dt, threads


def cpu_baseline(A, B, target_s: float, dtype="f16", epi=None, scales=(None, None)) -> dict:
    M, K = A.shape
    N = B.shape[0]
    rows, dt, threads = oracle_rows_timing(A, B, target_s, dtype=dtype, epi=epi, scales=scales)
    return {"value": metrics.tflops(rows, N, K, dt), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of D ({rows}x{N} outputs, K={K}) of the same seeded "
                      f"operands, fp64 accumulation, {dt:.2f} s"}


def workload_of(args):
    if args.shape:
        M, N, K = args.shape
        return inputs.Workload(f"shape_{M}x{N}x{K}", M, N, K, "normal:1/sqrtK", "normal:1/sqrtK", 99)
    return inputs.WORKLOADS[args.workload]


def operands_of(w, dtype="f16"):
    """(A, B, (a_scale, b_scale)); the scales (8-bit operands only) are None otherwise."""
    if dtype in FP8:
        if (w.K % 16) != 0:
            raise SystemExit(f"{w.name}: 8-bit rows of K = {w.K} bytes are not whole 16-byte units")
        A, B, sa, sb = inputs.operands_fp8(w.M, w.N, w.K, w.dist_a, w.dist_b, w.seed, fmt=dtype)
        return A, B, (sa, sb)
    if dtype == "bf16":
        return (*inputs.operands_bf16(w.M, w.N, w.K, w.dist_a, w.dist_b, w.seed), (None, None))
    return (*inputs.operands(w.M, w.N, w.K, w.dist_a, w.dist_b, w.seed), (None, None))


def out_dtype(dtype: str) -> str:
    return "f16" if dtype == "f16" else "bf16"


def in_bytes(dtype: str) -> int:
    return 1 if dtype in FP8 else 2


EPI_ALPHA, EPI_BETA = 1.5, 0.5


def epilogue_inputs(w, dtype="f16"):
    """C [M, N] and bias [N] of the fused-epilogue timing, uniform(-1, 1), seeded."""
    drawf = inputs.draw_bf16 if out_dtype(dtype) == "bf16" else inputs.draw
    return drawf(w.M, w.N, "uniform", w.seed + 2000), drawf(1, w.N, "uniform", w.seed + 3000).reshape(w.N)


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    w = workload_of(args)
    A, B, scales = operands_of(w, args.dtype)
    import oracle
    threads = oracle.default_threads()
    fn = oracle_rows_fn(A, B, args.dtype, epilogue_inputs(w, args.dtype) if args.epilogue else None, scales)
    # bound the whole run to a few minutes: size each step's sample of rows
    budget = 120.0
    per_step = max(0.05, min(2.0, budget / max(1, args.steps + args.warmup)))
    t = time.perf_counter()
    fn(0, 1, threads)
    one = max(time.perf_counter() - t, 1e-4)
    rows = int(max(1, min(w.M, per_step / one)))
    for i in range(args.warmup):
        r0 = (i * rows) % max(1, w.M - rows + 1)
        fn(r0, r0 + rows, threads)
    times = []
    for i in range(args.steps):
        r0 = (i * rows) % max(1, w.M - rows + 1)
        t = time.perf_counter()
        fn(r0, r0 + rows, threads)
        times.append(time.perf_counter() - t)
    sec = sum(times) / len(times)
    value = metrics.tflops(rows, w.N, w.K, sec)
    line = {
        "impl": "reference", "metric": metric_of(args.dtype), "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "operands": args.dtype,
                   "epilogue": (f"relu({EPI_ALPHA} * A·Bᵀ + {EPI_BETA} * C + bias)" if args.epilogue else "none"),
                   "sample_rows_per_step": rows, "note": "CPU oracle on a bounded sample of rows"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{rows} rows of D per step ({rows}x{w.N} outputs, K={w.K})"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(args, w, g, lib, dev, stream, pg, world, to_torch, tdt, dtype_code, A_h, B_h, C_h, bias_h,
            alpha=1.0, scale_h=None):
    """End to end through the C ABI from pinned host memory: every step copies
    its inputs host -> device, runs the GEMM and copies D back.  Steps are
    pipelined the way a caller would run them: inputs of step s+1 travel on a
    copy-in stream and D of step s-1 on a copy-out stream while step s
    computes, with two sets of device buffers; every step's copies are inside
    the timed region."""
    import torch

    def pinned(x):
        return to_torch(x).pin_memory()

    host_in = [pinned(A_h), pinned(B_h)]
    if args.epilogue:
        host_in += [pinned(C_h), pinned(bias_h)]
    if scale_h is not None:
        host_in.append(pinned(scale_h))               # the per-column scales are inputs too
    D_pin = [torch.empty((w.M, w.N), dtype=tdt).pin_memory() for _ in range(2)]
    bufs = [[torch.empty_like(h, device=dev) for h in host_in] for _ in range(2)]
    D_dev = [torch.empty((w.M, w.N), dtype=tdt, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    epis = []
    for b in range(2):
        sc = bufs[b][-1].data_ptr() if scale_h is not None else None
        if args.epilogue:
            epis.append(g.Epilogue(alpha * EPI_ALPHA, EPI_BETA, bufs[b][2].data_ptr(), bufs[b][3].data_ptr(),
                                   int(g.Activation.RELU), 0, sc))
        elif scale_h is not None:
            epis.append(g.Epilogue(alpha, 0.0, None, None, 0, 0, sc))
        else:
            epis.append(None)

    def launch(b):
        a, bb, d = bufs[b][0].data_ptr(), bufs[b][1].data_ptr(), D_dev[b].data_ptr()
        h = stream.cuda_stream
        if epis[b] is not None:
            st = lib.gemm_nt_ex(dtype_code, a, bb, d, w.M, w.N, w.K, g.ctypes.byref(epis[b]), 0, h)
        elif args.dtype == "bf16":
            st = lib.gemm_bf16_nt(a, bb, d, w.M, w.N, w.K, h)
        else:
            st = lib.gemm_f16_nt(a, bb, d, w.M, w.N, w.K, h)
        if st != 0:
            raise g.GemmError(st, "e2e launch")

    def run(n_steps, first):
        for k in range(n_steps):
            step_i = first + k
            b = step_i % 2
            if step_i >= 2:
                s_in.wait_event(ev_comp[b])       # buffer b's inputs no longer read
            with torch.cuda.stream(s_in):
                for dst, src in zip(bufs[b], host_in):
                    dst.copy_(src, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if step_i >= 2:
                stream.wait_event(ev_out[b])      # D of step s-2 copied out
            launch(b)
            ev_comp[b].record(stream)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                D_pin[b].copy_(D_dev[b], non_blocking=True)
                ev_out[b].record(s_out)

    e2e_steps = max(3, min(args.steps, 20))
    run(2, 0)
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    stream.wait_event(e0)
    s_out.wait_event(e0)
    run(e2e_steps, 2)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(pg, e2e_ms, dev)
    g.gemm_f16_nt_check(stream=stream, device=dev)
    return {"value": job_tflops(world, w.M, w.N, w.K, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
            "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host_in),
            "d2h_bytes_per_step": D_pin[0].numel() * D_pin[0].element_size(),
            "pipelining": "inputs of the next step and D of the previous one move on their own "
                          "streams while a step computes (two buffer sets)"}


# ---------------------------------------------------------------- the other workloads
def rotated_copies(torch, dev, A, B, min_bytes: int = L2_ROTATE_BYTES):
    """[(a_ptr, b_ptr)] of enough copies of A and B, packed in one buffer, that
    launches rotating over them never find their operands in L2 (a single copy
    when A and B already exceed min_bytes).  Returns (pointers, buffer)."""
    per_a, per_b = A.numel(), B.numel()
    ab_bytes = (per_a + per_b) * A.element_size()
    if ab_bytes >= min_bytes:
        return [(A.data_ptr(), B.data_ptr())], (A, B)
    stride = -(-(per_a + per_b) // 128) * 128          # 256-byte aligned copies
    copies = max(4, -(-min_bytes // (stride * A.element_size())))
    buf = torch.empty((copies, stride), dtype=A.dtype, device=dev)
    buf[:, :per_a].copy_(A.reshape(1, -1).expand(copies, -1))
    buf[:, per_a:per_a + per_b].copy_(B.reshape(1, -1).expand(copies, -1))
    base, esz = buf.data_ptr(), A.element_size()
    return [(base + c * stride * esz, base + (c * stride + per_a) * esz) for c in range(copies)], buf


def time_workload(args, g, lib, dev, stream, w, peaks) -> dict:
    """One named fp16 workload through gemm_f16_nt (AUTO), timed the way the
    headline is: warm-up launches, then back-to-back launches between one CUDA
    event pair on the launch stream, operands rotated past L2."""
    import torch
    A_h, B_h = inputs.operands(w.M, w.N, w.K, w.dist_a, w.dist_b, w.seed)
    A, B = torch.from_numpy(A_h).to(dev), torch.from_numpy(B_h).to(dev)
    D = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    ptrs, keep = rotated_copies(torch, dev, A, B)
    plan = g.gemm_f16_nt_plan(w.M, w.N, w.K)
    h, d_ptr, n_copies = stream.cuda_stream, D.data_ptr(), len(ptrs)
    cur = [0]

    def step():
        a, b = ptrs[cur[0]]
        cur[0] = (cur[0] + 1) % n_copies
        st = lib.gemm_f16_nt(a, b, d_ptr, w.M, w.N, w.K, h)
        if st != 0:
            raise g.GemmError(st, f"gemm_f16_nt {w.name}")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a short pilot run sizes the timed region to at least ~2 ms of launches
    e0.record(stream)
    for _ in range(10):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    pilot_ms = e0.elapsed_time(e1) / 10
    n = int(min(20000, max(args.steps, math.ceil(2.0 / max(pilot_ms, 1e-4)))))
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    g.gemm_f16_nt_check(stream=stream, device=dev)
    ms = e0.elapsed_time(e1) / n
    tf = metrics.tflops(w.M, w.N, w.K, ms * 1e-3)
    rec = {"M": w.M, "N": w.N, "K": w.K, "variant": plan["variant"], "grid_ctas": plan["grid_ctas"],
           "launches": n, "ms_per_launch": ms, "value": tf, "unit": UNIT,
           "l2": (f"A and B rotated over {n_copies} copies ({n_copies * (A.numel() + B.numel()) * 2 >> 20} MiB)"
                  if n_copies > 1 else "inputs larger than L2")}
    peak = float(peaks["bf16_tflops"]) if peaks and peaks.get("bf16_tflops") else FALLBACK_PEAK_TFLOPS
    if plan["variant"] == "SKINNY_SPLITK":
        hbm = float(peaks["hbm_gbs"]) if peaks and peaks.get("hbm_gbs") else 6800.0
        gbs = metrics.gbs(metrics.compulsory_bytes(w.M, w.N, w.K), ms * 1e-3)
        rec["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm}
    else:
        rec["roofline"] = {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak}
    del keep
    return rec


# ---------------------------------------------------------------- GPU leg
def run_ours(args):
    import torch
    import dense_fp16_gemm_f16_gb300 as g
    from dense_fp16_gemm_f16_gb300 import build as gbuild

    rank, local_rank, world = dist_env()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    # one process builds (ranks would otherwise race on the same output files)
    if local_rank == 0:
        gbuild.build()
    if pg:
        pg.barrier()
    g.load()
    w = workload_of(args)
    A_h, B_h, (a_scale, b_scale_h) = operands_of(w, args.dtype)
    tdt = torch.bfloat16 if out_dtype(args.dtype) == "bf16" else torch.float16
    dtype_code = int({"f16": g.Dtype.F16, "bf16": g.Dtype.BF16, "e4m3": g.Dtype.E4M3,
                      "e5m2": g.Dtype.E5M2}[args.dtype])

    def to_torch(x):
        # bf16 values travel as uint16 bit patterns, 8-bit operands as uint8
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(x)

    stream = torch.cuda.Stream(device=dev)
    A = to_torch(A_h).to(dev)
    B = to_torch(B_h).to(dev)
    D = torch.empty((w.M, w.N), dtype=tdt, device=dev)
    plan = g.gemm_nt_plan_ex(dtype_code, w.M, w.N, w.K)
    lib = g.load()
    s_handle = stream.cuda_stream
    # Operands smaller than twice the L2 are rotated over enough copies that
    # consecutive launches never find them in L2 (no flush needed between them).
    ab_bytes = (w.M * w.K + w.N * w.K) * in_bytes(args.dtype)
    copies = 1 if ab_bytes >= L2_ROTATE_BYTES else max(4, min(64, -(-L2_ROTATE_BYTES // max(ab_bytes, 1))))
    As, Bs = [A], [B]
    for _ in range(copies - 1):
        As.append(A.clone())
        Bs.append(B.clone())
    a_ptrs = [t.data_ptr() for t in As]
    b_ptrs = [t.data_ptr() for t in Bs]
    d_ptr = D.data_ptr()
    cur = [0]
    C_h = bias_h = C = bias = None
    # 8-bit operands: the per-tensor scale of A is alpha, B's per-row scales scale D's columns
    alpha = float(np.float32(a_scale)) if a_scale is not None else 1.0
    scale_n = torch.from_numpy(b_scale_h).to(dev) if b_scale_h is not None else None
    sc_ptr = scale_n.data_ptr() if scale_n is not None else None
    if args.epilogue:
        C_h, bias_h = epilogue_inputs(w, args.dtype)
        C, bias = to_torch(C_h).to(dev), to_torch(bias_h).to(dev)
        epi = g.Epilogue(alpha * EPI_ALPHA, EPI_BETA, C.data_ptr(), bias.data_ptr(), int(g.Activation.RELU), 0,
                         sc_ptr)
        epi_ref = g.ctypes.byref(epi)
    elif scale_n is not None:
        epi = g.Epilogue(alpha, 0.0, None, None, 0, 0, sc_ptr)
        epi_ref = g.ctypes.byref(epi)

    if args.epilogue or scale_n is not None:
        def step():
            i = cur[0] = (cur[0] + 1) % copies
            st = lib.gemm_nt_ex(dtype_code, a_ptrs[i], b_ptrs[i], d_ptr, w.M, w.N, w.K, epi_ref, 0, s_handle)
            if st != 0:
                raise g.GemmError(st, "gemm_nt_ex")
    elif args.dtype == "bf16":
        def step():
            i = cur[0] = (cur[0] + 1) % copies
            st = lib.gemm_bf16_nt(a_ptrs[i], b_ptrs[i], d_ptr, w.M, w.N, w.K, s_handle)
            if st != 0:
                raise g.GemmError(st, "gemm_bf16_nt")
    else:
        def step():
            i = cur[0] = (cur[0] + 1) % copies
            st = lib.gemm_f16_nt(a_ptrs[i], b_ptrs[i], d_ptr, w.M, w.N, w.K, s_handle)
            if st != 0:
                raise g.GemmError(st, "gemm_f16_nt")

    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    g.gemm_f16_nt_check(stream=stream, device=dev)

    # timed region: K launches back to back on `stream` between one event pair
    # (an event between launches would stop a launch overlapping the previous
    # kernel's tail, which the library allows)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if pg:
        pg.barrier()
    g.gemm_f16_nt_check(stream=stream, device=dev)
    region_ms = ev0.elapsed_time(ev1)
    ms_per_step = region_ms / args.steps
    launch_ms = ms_per_step          # average launch duration over the timed region (this rank)
    ms_per_step = max_over_ranks(pg, ms_per_step, dev)
    if sampler:
        sampler.mark(t_wall0, t_wall1)

    # Spread of the per-launch time: after the timed region, the same launches
    # in (up to) 30 batches with an event pair around each; reported beside the
    # value, which stays the one-region measurement above.
    # 30 batches of at least 1 ms each (more launches per batch than steps / 30
    # for launches under ~33 us); short diagnostic runs keep one launch per step
    batches = min(30, args.steps)
    per_batch = max(1, args.steps // batches)
    if batches == 30:
        per_batch = max(per_batch, math.ceil(1.0 / max(launch_ms, 1e-6)))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(batches + 1)]
    evs[0].record(stream)
    for b in range(batches):
        for _ in range(per_batch):
            step()
        evs[b + 1].record(stream)
    torch.cuda.synchronize(dev)
    g.gemm_f16_nt_check(stream=stream, device=dev)
    per_launch = sorted(evs[b].elapsed_time(evs[b + 1]) / per_batch for b in range(batches))
    spread = {"batches": batches, "launches_per_batch": per_batch, "batch_ms_min": per_launch[0] * per_batch,
              "median_ms": statistics.median(per_launch), "min_ms": per_launch[0],
              "p90_ms": per_launch[min(batches - 1, int(0.9 * batches))]}

    value = job_tflops(world, w.M, w.N, w.K, ms_per_step)

    # end to end through the C ABI: pinned host operands in, pinned host result out
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, g, lib, dev, stream, pg, world, to_torch, tdt, dtype_code, A_h, B_h, C_h, bias_h,
                      alpha, b_scale_h)

    # the other named workloads (fp16 plain product), same timing rules, and one
    # mid shape whose few tiles and long K loop take the split-K path
    configs = None
    if (not args.no_configs and rank == 0 and not args.shape and args.workload == inputs.HEADLINE
            and args.dtype == "f16" and not args.epilogue):
        peaks_c = measured_peaks()
        extra = [inputs.Workload("split_k_512x2048x8192", 512, 2048, 8192, "uniform", "uniform", 6)]
        configs = {wl.name: time_workload(args, g, lib, dev, stream, wl, peaks_c)
                   for wl in list(inputs.WORKLOADS.values()) + extra if wl.name != inputs.HEADLINE}

    clocks = sampler.stop() if sampler else None
    if pg:
        pg.barrier()
    if rank != 0:
        pg.destroy_process_group()
        return 0

    peaks = measured_peaks()
    # dense fp16 and bf16 tensor rates are the same on this architecture (ratio 1);
    # the dense fp8 rate is twice that (nominal 4.5 against 2.25 PFLOP/s)
    ratio = 2.0 if args.dtype in FP8 else 1.0
    if peaks and peaks.get("bf16_tflops"):
        peak = float(peaks["bf16_tflops"]) * ratio
        peak_src = ("measured bf16 cuBLAS burst x 2 (nominal dense fp8 : bf16 ratio)" if ratio != 1.0 else
                    "measured (bf16 cuBLAS burst, fp16 rate = bf16 rate)")
    else:
        peak = FALLBACK_PEAK_TFLOPS * ratio
        peak_src = "fallback" + (" x 2 (nominal dense fp8 : bf16 ratio)" if ratio != 1.0 else "")
    achieved = metrics.tflops(w.M, w.N, w.K, launch_ms * 1e-3)
    # the ncu counters were taken on the plain product (fp16), and for 8-bit
    # operands on the product with their scales
    traffic = None
    if not args.epilogue:
        traffic = recorded_traffic(w.name if args.dtype == "f16" else f"{w.name}/{args.dtype}")
    if plan["variant"] == "SKINNY_SPLITK":
        hbm = float(peaks["hbm_gbs"]) if peaks and peaks.get("hbm_gbs") else 6800.0
        # algorithmic bytes: A and B read once, D written once (+ C and bias read with the
        # epilogue, + the per-column scales of 8-bit operands)
        alg_bytes = ((w.M * w.K + w.N * w.K) * in_bytes(args.dtype) + w.M * w.N * 2
                     + (w.M * w.N * 2 + w.N * 2 if args.epilogue else 0) + (w.N * 4 if b_scale_h is not None else 0))
        gbs = metrics.gbs(alg_bytes, launch_ms * 1e-3)
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "traffic": traffic, "peak_source": "measured" if peaks else "fallback"}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src}
        if peaks and peaks.get("bf16_tflops_sustained"):
            # context: the same against the measured sustained rate (seconds of
            # back-to-back cuBLAS under the power cap), which long runs approach
            roofline["frac_of_sustained"] = achieved / (float(peaks["bf16_tflops_sustained"]) * ratio)

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(A_h, B_h, args.cpu_seconds, args.dtype, (C_h, bias_h) if args.epilogue else None,
                           (a_scale, b_scale_h))

    line = {
        "metric": metric_of(args.dtype), "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "accumulate": "f32",
                   "output": out_dtype(args.dtype),
                   "scales": ("A per tensor (alpha), B per row (per-column scale of D), fp32" if b_scale_h is not None
                              else "none"),
                   "epilogue": (f"relu({EPI_ALPHA} * A·Bᵀ + {EPI_BETA} * C + bias)" if args.epilogue else "none"),
                   "variant": plan["variant"], "grid_ctas": plan["grid_ctas"],
                   "l2": (f"inputs larger than L2 (A+B = {ab_bytes >> 20} MiB >= {L2_ROTATE_BYTES >> 20} MiB); no flush"
                          if copies == 1 else
                          f"A and B rotated over {copies} copies ({copies * ab_bytes >> 20} MiB, > 2x the 129 MB L2) "
                          "so no launch finds its operands in L2; no flush"
                          if copies * ab_bytes >= L2_ROTATE_BYTES else
                          f"A and B rotated over {copies} copies ({copies * ab_bytes / 2**20:.1f} MiB), still within "
                          "L2: a warm-L2 number"),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "timing": "one CUDA event pair around the K back-to-back launches on the launch stream"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "per_launch_spread": spread,
        "configs": configs,
        "clocks": clocks,
        "device": device_info(local_rank),
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
