#!/usr/bin/env python3
"""Benchmark of the GB300 tensor-core GEMM C = epilogue(A . B).

One step = one C = epilogue(A . B) call over the workload's synthetic,
seeded inputs, already resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline] [--no-secondary]

Default workload: square8192_bf16 (bf16 M=N=K=8192, bf16 output), the
tensor-core roofline case.  Other workloads: see gemm_inputs.WORKLOADS.

Timing: W untimed warm-up steps; then K steps bracketed by a barrier and a
device synchronisation; each step's GEMM is timed with CUDA events on the
launching stream, and L2 is flushed between steps (outside the events) so
every step starts with a cold L2: by default a 256 MiB buffer is written and
a second 256 MiB buffer then read, so the write's dirty lines are written
back before the timed launch instead of during it (--flush write: the write
alone).  `value` is the whole-job
throughput: total FLOPs of all ranks / max-over-ranks of the summed event
time.  With N > 1 every rank runs an independent replica (the path has no
exchange step; "weak" scaling).

`--impl reference` times the CPU oracle (the plain fp64 triple loop) on the
host cores, on a bounded row-block sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gemm_inputs  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s of HBM3e the skinny-K target is stated against
# The only timing on the pages: a whole 4K denoiser frame (11 Swin layers,
# not one GEMM), on hardware the page does not name.  Context, not a target.
PAGES_CONTEXT = {"what": "whole 3840x2160 denoiser frame: isolated native phase-8 splice vs translated body",
                 "ms": {"splice": 14.90, "translated": 6.59}, "hardware": "not named on the page",
                 "source": "d4r, rrswin_enc2_epilogues.md (page header)",
                 "note": "context only: a whole-frame time of another engine, not comparable to one GEMM"}
METRIC = "GEMM TFLOP/s and % of GB300 dense fp16/bf16 peak (HBM GB/s for skinny-K)"
DEFAULT_WORKLOAD = "square8192_bf16"
HBM_BOUND = {"swin4k_proj_f16", "swin4k_backproj_f16", "swin4k_proj_i8w"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(gemm_inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg (profiling runs)")
    ap.add_argument("--no-secondary", action="store_true", help="skip the other-workload summary")
    ap.add_argument("--no-library-reference", action="store_true",
                    help="skip the same-run torch.matmul (cuBLAS) reference of tensor-bound workloads")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    ap.add_argument("--tune", action="store_true",
                    help="tune the launch configuration first (sg_tune) instead of the planner's heuristic")
    ap.add_argument("--flush", default="write+read", choices=["write+read", "write"],
                    help="L2 flush between timed steps: a 256 MiB write then a 256 MiB read (clean cold L2), "
                         "or the write alone (its dirty lines are written back during the timed launch)")
    ap.add_argument("--block-n", type=int, default=0, help="sg_config.block_n (0: the planner's)")
    ap.add_argument("--mode", type=int, default=0, help="sg_config.mode (0: the planner's)")
    ap.add_argument("--group-m", type=int, default=0, help="sg_config.group_m, the raster group (0: the planner's)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the CUDA sources with comments and whitespace removed, so that
    it changes only when the compiled code can."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_core_gemm_tma_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name)) as f:
                code = f.read()
            code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)           # block comments
            code = re.sub(r'//[^\n]*', " ", code)                            # line comments
            code = "".join(code.split())
            h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    cur = kernel_source_hash()
    with open(p) as f:
        for line in f:
            parts = line.split("#")[0].split()
            if len(parts) >= 3 and parts[0] == workload and parts[1] == cur:
                return int(float(parts[2]))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"sg_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples under load: the upper part of the clock distribution
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def device_inputs(w, device):
    """Host tensors of the workload's operands: (A, B, bias, R)."""
    import torch
    a, bias, r = w.a_bits(), w.bias(), w.r_bits()
    if w.in_dtype == "e4m3":
        A = torch.from_numpy(a).view(torch.float8_e4m3fn)
        B = torch.from_numpy(w.b_bits()).view(torch.float8_e4m3fn)
    else:
        tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[w.in_dtype]
        A = torch.from_numpy(a.view(np.int16)).view(tdt)
        if w.b_coded:  # (int8 codes, per-column fp32 scales)
            q, sc = w.b_codes()
            B = (torch.from_numpy(q), torch.from_numpy(sc))
        else:
            B = torch.from_numpy(w.b_bits().view(np.int16)).view(tdt)
    bias_t = None if bias is None else torch.from_numpy(bias.copy())
    R = None
    if r is not None:
        R = torch.from_numpy(r.view(np.int32 if w.out_dtype == "f32" else np.int16)).view(out_torch_dtype(w))
    return A, B, bias_t, R


def out_torch_dtype(w):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.out_dtype]


def time_steps(call, steps, stream, flush):
    """Per-step CUDA-event durations (ms) of `call`, with an L2 flush between."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in evs:
        flush()
        s.record(stream)
        call()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def b_operand(w):
    """B as the oracle takes it: bit patterns, or (int8 codes, scales)."""
    return w.b_codes() if w.b_coded else w.b_bits()


def oracle_rows(w, a, b, bias, r, rows, threads):
    """The oracle (as it stands) on rows 0..rows-1 of the workload."""
    import oracle
    if w.b_coded:
        q, s = b
        return oracle.gemm_qb(a[:rows], q, s, w.in_dtype, w.out_dtype, w.epilogue, bias, threads=threads)
    return oracle.gemm(a[:rows], b, w.in_dtype, w.out_dtype, w.epilogue, bias, threads=threads,
                       R_bits=None if r is None else r[:rows], r_dtype=w.out_dtype if r is not None else None)


def cpu_baseline_entry(w, target_s):
    """The oracle (as it stands) timed on the host cores on a row-block
    sample of the workload, as a cpu_baseline object."""
    dt, rows, flops, threads = cpu_oracle_sample(w, target_s=target_s)
    d = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
         "sample": f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} product ({rows * w.N} outputs, {dt:.2f} s)",
         "extrapolated": rows < w.M, "seconds": dt}
    if w.name in HBM_BOUND:
        d["gbs"] = w.algorithmic_bytes * rows / w.M / dt / 1e9
    return d


def call_latency(sg, w, device, stream, calls=200):
    """Per-call latency of a launch-bound product: the device time of back to
    back launches (no flush), the host time per stage_gemm call (the ctypes
    call and the launch, synchronised once at the end), and one
    host-buffer call (stage_gemm_host: copies in, GEMM, copy out) end to end."""
    import torch
    A_h, B_h, bias_h, R_h = device_inputs(w, device)
    A, B = A_h.to(device), B_h.to(device)
    C = torch.empty((w.M, w.N), dtype=out_torch_dtype(w), device=device)
    with torch.cuda.stream(stream):
        for _ in range(20):
            sg.stage_gemm(A, B, epilogue=w.epilogue, out=C, stream=stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(calls):
            sg.stage_gemm(A, B, epilogue=w.epilogue, out=C, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        host_us = (time.perf_counter() - t0) / calls * 1e6
        dev_us = e0.elapsed_time(e1) / calls * 1e3
        A_p, B_p = A_h.pin_memory(), B_h.pin_memory()
        out_h = torch.empty((w.M, w.N), dtype=out_torch_dtype(w), pin_memory=True)
        for _ in range(5):
            sg.stage_gemm_host(A_p, B_p, out_dtype=out_h.dtype, epilogue=w.epilogue, device=device, stream=stream,
                               out_host=out_h)
        torch.cuda.synchronize()
        ts = []
        for _ in range(50):
            t0 = time.perf_counter()
            sg.stage_gemm_host(A_p, B_p, out_dtype=out_h.dtype, epilogue=w.epilogue, device=device, stream=stream,
                               out_host=out_h)
            stream.synchronize()
            ts.append((time.perf_counter() - t0) * 1e6)
    return {"device_us_per_launch_back_to_back": dev_us, "host_us_per_call_back_to_back": host_us,
            "host_buffer_call_us_median": statistics.median(ts),
            "how": f"{calls} back-to-back stage_gemm calls on resident operands (CUDA events; host wall clock); "
                   "50 synchronised stage_gemm_host calls on pinned buffers (copies in and out included)"}


def cpu_oracle_sample(w, target_s=12.0, a=None, b=None, bias=None):
    """Time the oracle (as it stands) on a row-block sample of the workload:
    returns (seconds, rows, flops, threads)."""
    a = w.a_bits() if a is None else a
    b = b_operand(w) if b is None else b
    bias = w.bias() if bias is None else bias
    r = w.r_bits()
    threads = os.cpu_count() or 1
    rows = min(w.M, max(threads, 16))
    while True:
        t0 = time.perf_counter()
        oracle_rows(w, a, b, bias, r, rows, threads)
        dt = time.perf_counter() - t0
        if dt >= target_s / 4 or rows >= w.M:
            break
        rows = min(w.M, max(rows * 2, int(rows * (target_s / 2) / max(dt, 1e-3))))
    return dt, rows, 2.0 * rows * w.N * w.K, threads


def run_reference(args, w, rank, world):
    """The oracle arm: rank 0 only, on the host cores."""
    if rank != 0:
        return
    a, b, bias, r = w.a_bits(), b_operand(w), w.bias(), w.r_bits()
    # size one step's sample from a calibration run
    _, rows, _, threads = cpu_oracle_sample(w, target_s=4.0, a=a, b=b, bias=bias)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle_rows(w, a, b, bias, r, rows, threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    flops = 2.0 * rows * w.N * w.K
    tot = sum(times)
    value = flops * len(times) / tot / 1e12
    sample = f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} product per step ({rows * w.N} outputs)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, None),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, plan, flush_mode="write+read"):
    how = {"write+read": "a 256 MiB write then a 256 MiB read", "write": "a 256 MiB write"}[flush_mode]
    c = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "in_dtype": w.in_dtype, "out_dtype": w.out_dtype,
         "epilogue": w.epilogue, "accumulate": "f32", "layout": "A, B, C row-major, dense",
         "l2": f"flushed between timed steps ({how}, outside the timed events)",
         "description": w.description}
    if plan:
        rows = plan["block_m"] * (2 if plan.get("pair_mma") else 1)
        c["tile"] = f"{rows}x{plan['block_n']}x{plan['block_k']}"
        c["stages"] = plan["stages"]
        c["grid"] = plan["grid"]
        c["kernel_mode"] = {1: "single CTA", 3: "paired MMA (cta_group::2)",
                            6: "paired MMA over 256x512 tiles, two 256-column accumulators (cta_group::2)",
                            4: "resident B (one CTA per row tile, all of B in shared memory)",
                            5: "decoded panel (int8-coded B decoded once per CTA into the resident shared-memory "
                               "panel)"}.get(plan.get("mode"))
        c["raster_group_m"] = plan.get("group_m")
        c["tuned"] = plan.get("tuned", False)
    return c


def make_flush(device, mode):
    """The L2 flush run between timed steps (outside the events)."""
    import torch
    wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    if mode == "write":
        return lambda: wbuf.fill_(1)
    rbuf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def flush():
        wbuf.fill_(1)
        rbuf.sum()          # reads 256 MiB: the write's dirty lines leave L2 here
    return flush


def measure(sg, w, device, stream, steps, warmup, stages, inputs=None, tune=True, config=None,
            flush_mode="write+read"):
    import torch
    A_h, B_h, bias_h, R_h = inputs if inputs is not None else device_inputs(w, device)
    A = A_h.to(device)
    B = tuple(x.to(device) for x in B_h) if w.b_coded else B_h.to(device)
    bias = None if bias_h is None else bias_h.to(device)
    R = None if R_h is None else R_h.to(device)
    C = torch.empty((w.M, w.N), dtype=out_torch_dtype(w), device=device)
    if tune and config is None and stages == 0 and R is None and not w.b_coded:
        # the library's own tuner picks the configuration (outside the timed steps)
        sg.tune(A, B, epilogue=w.epilogue, bias=bias, out=C, stream=stream)
    flush = make_flush(device, flush_mode)

    def call():
        if w.b_coded:
            sg.stage_gemm_qb(A, B[0], B[1], epilogue=w.epilogue, bias=bias, stages=stages, out=C, stream=stream)
        else:
            sg.stage_gemm(A, B, epilogue=w.epilogue, bias=bias, stages=stages, out=C, stream=stream, residual=R,
                          config=config)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush()
            call()
        torch.cuda.synchronize()
        times = time_steps(call, steps, stream, flush)
    st = sg.device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed steps")
    return times, (A_h, B_h, bias_h, R_h), (A, B, bias, C)


def measure_e2e(sg, w, host_inputs, device, stream, steps, stages):
    """The same metric through the host-buffer API: pinned A, B (bias) copied
    in, C copied out, every step, timed with events on the stream."""
    import torch
    A_h, B_h, bias_h, R_h = host_inputs
    A_p = A_h.pin_memory()
    B_p = B_h.pin_memory()
    bias_p = None if bias_h is None else bias_h.pin_memory()
    R_p = None if R_h is None else R_h.pin_memory()
    out_h = torch.empty((w.M, w.N), dtype=out_torch_dtype(w), pin_memory=True)

    def call():
        sg.stage_gemm_host(A_p, B_p, out_dtype=out_h.dtype, epilogue=w.epilogue, bias_host=bias_p, stages=stages,
                           device=device, stream=stream, out_host=out_h, residual_host=R_p)

    with torch.cuda.stream(stream):
        call()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for s, e in evs:
            s.record(stream)
            call()
            e.record(stream)
        torch.cuda.synchronize()
    ms = [s.elapsed_time(e) for s, e in evs]
    h2d = A_p.numel() * A_p.element_size() + B_p.numel() * B_p.element_size()
    if bias_p is not None:
        h2d += bias_p.numel() * 4
    if R_p is not None:
        h2d += R_p.numel() * R_p.element_size()
    d2h = out_h.numel() * out_h.element_size()
    return sum(ms) / len(ms), h2d, d2h


def max_over_ranks(value: float, pg=None, device=None) -> float:
    """The largest of every rank's `value` (the job is as slow as its slowest
    replica).  With no process group: the value itself."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, world: int, steps: int, max_sum_ms: float) -> float:
    """Every rank runs the same workload (replicas): total FLOPs of all
    ranks over the slowest rank's summed step time."""
    return flops_per_step * world * steps / (max_sum_ms * 1e-3) / 1e12


def dram_reference(device, nbytes_write: int, steps: int = 10, flush_mode="write+read"):
    """Same-run DRAM references for an HBM-bound workload: a device memset
    of the workload's output bytes (write only) and a device-to-device copy
    of as many bytes (read + write), each timed like the GEMM (L2 flushed
    before each step, CUDA events).  Returns GB/s figures."""
    import torch
    n = (nbytes_write + 1) // 2
    x = torch.empty(n, dtype=torch.float16, device=device)
    y = torch.empty(n, dtype=torch.float16, device=device)
    flush = make_flush(device, flush_mode)

    def med(fn):
        for _ in range(2):
            fn()
        ts = []
        for _ in range(steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)
    w_ms = med(lambda: x.zero_())
    c_ms = med(lambda: y.copy_(x))
    return {"write_only_gbs": 2 * n / (w_ms * 1e-3) / 1e9, "copy_gbs": 4 * n / (c_ms * 1e-3) / 1e9,
            "bytes": 2 * n, "how": "cudaMemsetAsync of the output's bytes; device copy of as many bytes (read+write)"}


def library_reference(w, dev_tensors, stream, steps=10, warmup=3, flush_mode="write+read"):
    """Same-run library reference for a tensor-bound fp16/bf16 workload: the
    same product through torch.matmul (cuBLAS) plus torch's own ReLU / bias
    ops for the epilogue, on the same device tensors, timed like the GEMM (L2
    flushed before each step, CUDA events).  Context only: it is not the
    product path and not the driver's reference arm."""
    import torch
    if w.name in HBM_BOUND or w.dist_r is not None or w.b_coded:
        return None
    A, B, bias, C = dev_tensors
    flush = make_flush(A.device, flush_mode)
    if w.in_dtype == "e4m3":
        # cuBLAS FP8 through torch._scaled_mm: unit scales, fp32 accumulation
        # (use_fast_accum=False), B column-major as it requires (laid out
        # once, outside the timed steps)
        if w.epilogue != "none" or not hasattr(torch, "_scaled_mm"):
            return None
        Bc = B.t().contiguous().t()
        one = torch.ones((), dtype=torch.float32, device=A.device)

        def call():
            torch._scaled_mm(A, Bc, scale_a=one, scale_b=one, out_dtype=C.dtype, use_fast_accum=False)
        impl = "torch._scaled_mm (cuBLAS FP8, fp32 accumulation)"
    else:
        # torch's matmul writes the operands' type only: an fp32-output
        # product is timed with fp16/bf16 output (the library's nearest form)
        Cl = C if C.dtype == A.dtype else torch.empty(C.shape, dtype=A.dtype, device=A.device)

        def call():
            if w.epilogue == "bias_relu":
                torch.addmm(bias.to(Cl.dtype), A, B, out=Cl)
            else:
                torch.matmul(A, B, out=Cl)
            if w.epilogue != "none":
                Cl.relu_()
        impl = "torch.matmul (cuBLAS)" + (" + torch ReLU" if w.epilogue != "none" else "")
        if Cl is not C:
            impl += f" with {str(A.dtype).replace('torch.', '')} output (torch has no fp32-output form)"

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush()
            call()
        torch.cuda.synchronize()
        times = time_steps(call, steps, stream, flush)
    ms = sum(times) / len(times)
    return {"impl": impl, "value": w.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms}


def roofline_of(w, ms, peaks, traffic, library=None):
    """The dominant (only) kernel's roofline.  `frac` is against the measured
    peak; for a tensor-bound workload with a same-run library figure,
    `frac_conservative` is against the larger of the two (a library kernel
    that beats the measured peak makes that the honest denominator); an
    HBM-bound one also gets its fraction of the nominal ~8 TB/s."""
    if w.name in HBM_BOUND:
        achieved = w.algorithmic_bytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": f"{peaks['source']} hbm_gbs (copy bandwidth)",
                "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                "algorithmic_bytes_per_launch": w.algorithmic_bytes}
    achieved = w.flops / (ms * 1e-3) / 1e12
    # fp16 and bf16 dense tensor rates are the same (nominal ratio 1); FP8 is
    # twice the bf16 rate (nominal 4.5 vs 2.25 PFLOP/s dense)
    ratio = 2.0 if w.in_dtype == "e4m3" else 1.0
    peak = peaks["bf16_tflops"] * ratio
    src = f"{peaks['source']} bf16_tflops (burst; kernel timed alone)"
    if ratio != 1.0:
        src += " x 2 (nominal FP8 : bf16 dense ratio)"
    r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
         "frac": achieved / peak, "traffic": traffic, "peak_source": src,
         "algorithmic_flops_per_launch": w.flops, "algorithmic_bytes_per_launch": w.algorithmic_bytes}
    if library is not None:
        denom = max(peak, library["value"])
        r["frac_conservative"] = achieved / denom
        r["frac_conservative_of"] = ("same-run library " + library["impl"]) if library["value"] > peak else \
            "measured peak (above the same-run library)"
    return r


def main():
    args = parse()
    rank, world, local = dist_env()
    w = gemm_inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import tensor_core_gemm_tma_gb300 as sg
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist
    sg.load_library()
    stream = torch.cuda.Stream(device)
    peaks = load_peaks()

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    barrier()
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    clocks = ClockSampler(cvd.split(",")[local] if cvd else local)
    host_inputs = device_inputs(w, device)
    cfg = None
    if args.block_n or args.mode or args.group_m:
        cfg = {"block_n": args.block_n, "mode": args.mode, "group_m": args.group_m}
    # warm-up + timed steps (the clock sampler runs over the timed region)
    with clocks:
        barrier()
        times, host_inputs, dev_tensors = measure(sg, w, device, stream, args.steps, args.warmup, args.stages,
                                                  inputs=host_inputs, tune=args.tune, config=cfg,
                                                  flush_mode=args.flush)
        barrier()
    sum_ms = max_over_ranks(sum(times), pg, device)
    ms = sum_ms / len(times)
    value = whole_job_tflops(w.flops, world, len(times), sum_ms)
    plan = sg.plan(w.M, w.N, w.K, host_inputs[0].dtype, out_torch_dtype(w), w.epilogue, args.stages,
                   config=None if w.b_coded else cfg)
    if w.b_coded:
        plan["mode"] = 5  # mode 4's geometry with the panel decoded from int8 codes (stage_gemm_qb)
    plan["tuned"] = args.tune and cfg is None and args.stages == 0 and w.dist_r is None

    lib_ref = None
    if rank == 0 and not args.no_library_reference:
        lib_ref = library_reference(w, dev_tensors, stream, flush_mode=args.flush)
        if lib_ref is not None:
            lib_ref["ours_over_library"] = (w.flops / (ms * 1e-3) / 1e12) / lib_ref["value"]

    e2e = None
    if not args.no_e2e and not w.b_coded:  # the host-buffer entry takes 16-bit or FP8 B only
        del dev_tensors
        e2e_ms, h2d, d2h = measure_e2e(sg, w, host_inputs, device, stream, max(3, min(args.steps, 10)), args.stages)
        e2e = {"value": w.flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "tensor_core_gemm_tma_gb300.stage_gemm_host -> sg_gemm_host (C ABI; pinned host buffers, row-chunked copies overlapped with the GEMMs)"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.in_dtype, "data": "synthetic (seeded SplitMix64, see gemm_inputs)",
        "config": config_of(w, plan, args.flush),
        "roofline": roofline_of(w, ms, peaks, recorded_traffic(w.name), lib_ref),
        "ms_per_step_min": min(times), "ms_per_step_median": statistics.median(times),
        "gpu_launches": len(times),
        "gpu_launches_note": "one stage_gemm kernel launch per timed step (the L2 flush between steps is torch "
                             "fill and sum kernels, outside the timed events)",
        "clocks": clocks.summary(),
        "e2e": e2e,
        "kernel_source_hash": kernel_source_hash(),
        "pages_context": PAGES_CONTEXT,
    }
    if lib_ref is not None:
        line["library_reference"] = lib_ref
    if w.name in HBM_BOUND:
        line["hbm_gbs"] = line["roofline"]["achieved"]
        out_bytes = w.M * w.N * {"f32": 4, "f16": 2, "bf16": 2}[w.out_dtype]
        line["dram_reference"] = dram_reference(device, out_bytes, flush_mode=args.flush)

    if rank == 0 and not args.no_secondary and args.workload == DEFAULT_WORKLOAD and cfg is None:
        line["secondary"] = secondaries(sg, device, stream, peaks, args)

    if rank == 0 and not args.no_cpu_baseline and world >= 1:
        line["cpu_baseline"] = cpu_baseline_entry(w, 12.0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


# The other workloads, each measured as the main one is (10 timed steps after
# 3 warm-up steps, L2 flushed between steps), with its own roofline, same-run
# library figure where there is one, and its own CPU-oracle baseline.  The
# 4096^3 ReLU product also runs in the pages' tiling (128 x 128 output tiles:
# one CTA per tile, and CTA pairs whose CTAs each own one 128 x 128 tile).
SECONDARY = ["square256_f16", "ragged1000_f16", "relu4096_f16", "swin4k_proj_f16", "swin4k_backproj_f16",
             "square8192_e4m3", "swin4k_proj_i8w"]
PAGES_TILINGS = [({"block_n": 128, "mode": 3}, "128x128 output tile per CTA, CTA pairs sharing B (paired MMA)"),
                 ({"block_n": 128, "mode": 1}, "128x128 output tile per CTA, one CTA per tile")]


def secondaries(sg, device, stream, peaks, args):
    out = []

    def one(ws, config=None, label=None):
        t, _, dt = measure(sg, ws, device, stream, 10, 3, 0, tune=args.tune, config=config, flush_mode=args.flush)
        m = sum(t) / len(t)
        lr = None if args.no_library_reference or config is not None else \
            library_reference(ws, dt, stream, flush_mode=args.flush)
        del dt
        p = sg.plan(ws.M, ws.N, ws.K, in_torch_dtype(ws), out_torch_dtype(ws), ws.epilogue, config=config) \
            if not ws.b_coded else None
        e = {"workload": ws.name, "ms_per_step": m, "TFLOP/s": ws.flops / (m * 1e-3) / 1e12,
             "roofline": roofline_of(ws, m, peaks, recorded_traffic(ws.name) if config is None else None, lr)}
        if p is not None:
            e["plan"] = {k: p[k] for k in ("block_m", "block_n", "mode", "pair_mma", "stages", "grid", "tiles")}
        if label:
            e["tiling"] = label
            e["config"] = config
        if lr is not None:
            lr["ours_over_library"] = e["TFLOP/s"] / lr["value"]
            e["library_reference"] = lr
        return e

    for name in SECONDARY:
        ws = gemm_inputs.WORKLOADS[name]
        e = one(ws)
        if name == "square256_f16":
            e["latency"] = call_latency(sg, ws, device, stream)
        if name in ("swin4k_proj_f16", "swin4k_proj_i8w"):
            e["pages_context"] = "see the line's pages_context (a whole-frame figure, not this GEMM)"
        if not args.no_cpu_baseline:
            e["cpu_baseline"] = cpu_baseline_entry(ws, 2.5)
        out.append(e)
        if name == "relu4096_f16":
            for config, label in PAGES_TILINGS:
                out.append(one(ws, config, label))
    return out


def in_torch_dtype(w):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}[w.in_dtype]


if __name__ == "__main__":
    main()
