#!/usr/bin/env python3
"""Throughput of the GB300 fp16 TN GEMM library on its measured workloads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one call of the library's public C entry point (gemm_tn_f16 or
gemm_tn_f16_batched) on one batch of synthetic input already resident in
HBM: every kernel of the hot path (operand repack, tensor-core GEMM, split-K
reduction, as the plan needs) runs inside it.  Rank 0 prints one JSON line.

- value: TFLOP/s of the whole job (2*M*N*K*batch per step, summed over ranks)
  over device time measured with CUDA events on the launching stream; between
  steps L2 is flushed by writing a 256 MiB buffer outside the timed events.
- roofline: the dominant (tensor-core GEMM) kernel's achieved TFLOP/s against
  the measured peak in MEASURED_PEAKS.json (bf16 cuBLAS; fp16 has the same
  nominal tensor rate): its sustained figure when the timed steps run back to
  back for half a second or more (the part then sits at its power cap), else
  its burst figure; plus the kernel's DRAM traffic from the committed ncu
  capture when that capture matches the current kernel sources.
- e2e: the same metric through the same C call with the inputs copied from
  pinned host memory and D copied back inside the timed region.
- cpu_baseline: the CPU oracle (fp64, test infrastructure) timed on this
  host's cores on a bounded sample of output rows of the same workload.
- per_config: the other measured workloads, timed the same way (shorter).
- --impl reference: the oracle alone, timed on the host cores, each step a
  bounded sample of rows of the same workload.

Multi-GPU: each rank runs the same problem on its own GPU (replicas, no
collective on the data path); a barrier brackets the timed region and the
slowest rank's time is used.
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
sys.path.insert(0, ROOT)

METRIC = "TFLOPS and % of GB300 dense FP16 peak per config (1 GPU), vs CPU oracle"
UNIT = "TFLOP/s"
MAIN_WORKLOAD = "gemm_8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# A timed region of back-to-back steps at least this long (seconds) is compared with the
# sustained tensor peak, a shorter one with the burst peak.
SUSTAINED_S = 0.5
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129e6


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(files):
    """Hash of the CUDA sources the captured kernel is built from (names under csrc/)."""
    h = hashlib.sha256()
    for name in sorted(files):
        with open(os.path.join(ROOT, "dense_fp16_gemm_tn_gb300", "csrc", name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_key):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu capture,
    or None when the capture is missing or was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload_key)
    try:
        if not e or e.get("kernel_source_hash") != kernel_source_hash(e["sources"]):
            return None
    except (KeyError, OSError):
        return None
    return e.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.15)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"],
                                 parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ device side

class Problem:
    """Device-resident operands for one workload (seeded torch RNG on the GPU)."""

    def __init__(self, w, device, seed):
        import torch
        self.w = w
        g = torch.Generator(device=device)
        g.manual_seed(seed)

        def make(rows, cols, ld, batch):
            shape = (batch, rows, ld)
            if w.dist == "uniform":
                x = torch.rand(shape, generator=g, device=device, dtype=torch.float32) * 2 - 1
            else:
                x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
            x = x.half()
            if ld > cols:
                x[:, :, cols:] = float("nan")
            return x.contiguous()

        self.A = make(w.M, w.K, w.lda_, w.batch)
        self.B = make(w.N, w.K, w.ldb_, w.batch)
        self.C = make(w.M, w.N, w.ldc_, w.batch) if w.beta != 0 else None
        self.D = torch.empty((w.batch, w.M, w.ldd_), dtype=torch.float16, device=device)
        self.sA, self.sB = w.M * w.lda_, w.N * w.ldb_
        self.sC, self.sD = w.M * w.ldc_, w.M * w.ldd_

    def call(self, G, stream, A=None, B=None, C=None, D=None):
        w = self.w
        A = self.A if A is None else A
        B = self.B if B is None else B
        C = self.C if C is None else C
        D = self.D if D is None else D
        if w.batch == 1:
            G.gemm_tn_f16(A, w.lda_, B, w.ldb_, C, w.ldc_, D, w.ldd_, w.M, w.N, w.K, w.alpha, w.beta, stream)
        else:
            G.gemm_tn_f16_batched(A, w.lda_, self.sA, B, w.ldb_, self.sB, C, w.ldc_, self.sC, D, w.ldd_, self.sD,
                                  w.M, w.N, w.K, w.batch, w.alpha, w.beta, stream)


def launches_per_step(G, w, sms):
    p = G.gemm_tn_f16_plan(w.M, w.N, w.K, w.batch, w.lda_, w.ldb_, w.ldc_, w.ldd_, w.M * w.lda_, w.N * w.ldb_,
                           w.M * w.ldc_, w.M * w.ldd_, w.beta, 15, sms)
    if p["kernel"] == 0:
        return 0, p
    if p["kernel"] == 1:
        return 1, p
    return 1 + p["pack_a"] + p["pack_b"] + (1 if p["splits"] > 1 else 0), p


def needs_flush(w):
    """L2 is flushed before every step unless the operands exceed twice its size
    (then they stream from HBM whatever the replacement policy keeps)."""
    return w.algorithmic_bytes < 2 * L2_BYTES


def flush_l2(flush_buf, read_buf, i):
    """Write 256 MiB (evicts L2), then read another 256 MiB so that the dirty lines
    of the write are written back here and not inside the next timed GEMM."""
    flush_buf.fill_(i & 0x7F)
    read_buf.sum(dtype=torch_int64())


def torch_int64():
    import torch
    return torch.int64


def time_steps(prob, G, steps, warmup, flush_buf, dist, read_buf=None):
    """Per-step device times (ms) of the GEMM call; L2 flushed before each step
    when the workload's operands fit in it."""
    import torch
    stream = torch.cuda.current_stream()
    flush = needs_flush(prob.w) and read_buf is not None
    for _ in range(warmup):
        prob.call(G, stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    dist_barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        if flush:
            flush_l2(flush_buf, read_buf, i)  # outside the events
        ev[i][0].record(stream)
        prob.call(G, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    dist_barrier(dist)
    return [a.elapsed_time(b) for a, b in ev], wall


def time_l2_hot(prob, G, steps):
    """Median device time of one call with its operands left in L2 by the previous call.
    A 50 us GPU-side delay (torch.cuda._sleep) before each event pair lets the host
    queue the call before the GPU reaches the first event, so the host's own call
    overhead stays outside the measured interval."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(3):
        prob.call(G, stream)
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        torch.cuda._sleep(100000)  # about 50 us at 2 GHz
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        prob.call(G, stream)
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median([a.elapsed_time(b) for a, b in ts])


def time_back_to_back(prob, G, n):
    """Device time per call of n calls queued back to back (operands in L2)."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(3):
        prob.call(G, stream)
    torch.cuda.synchronize()
    torch.cuda._sleep(4000000)  # about 2 ms: the host queues all n calls while the GPU waits
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        prob.call(G, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def time_e2e(prob, G, steps, warmup):
    """The same problem end to end from page-locked host buffers: every step copies A, B
    (and C) to the device and D back, inside the timed region.  A single GEMM goes
    through the library's host-buffer call (copies pipelined with the compute in row
    blocks); a batched one copies with torch and calls the device entry point."""
    import torch
    stream = torch.cuda.current_stream()
    w = prob.w
    hA = prob.A.cpu().pin_memory()
    hB = prob.B.cpu().pin_memory()
    hC = prob.C.cpu().pin_memory() if prob.C is not None else None
    hD = torch.empty(prob.D.shape, dtype=prob.D.dtype).pin_memory()
    if w.batch == 1:
        def step():
            G.gemm_tn_f16_host(hA, w.lda_, hB, w.ldb_, hC, w.ldc_, hD, w.ldd_, w.M, w.N, w.K, w.alpha, w.beta,
                               stream)
    else:
        dA, dB = torch.empty_like(prob.A), torch.empty_like(prob.B)
        dC = torch.empty_like(prob.C) if prob.C is not None else None
        dD = torch.empty_like(prob.D)

        def step():
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            if dC is not None:
                dC.copy_(hC, non_blocking=True)
            prob.call(G, stream, dA, dB, dC, dD)
            hD.copy_(dD, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # bytes that cross the link each step (matrix elements only)
    h2d = 2 * w.batch * (w.M * w.K + w.N * w.K + (w.M * w.N if w.beta != 0 else 0))
    d2h = 2 * w.batch * w.M * w.N
    return ms, h2d, d2h


def slowest_rank_ms(total_ms, dist, device=None):
    """The timed region's length on the slowest rank (replicas: the job ends with it)."""
    if dist is None:
        return total_ms
    import torch
    on = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([total_ms], device=on, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_step, steps, total_ms):
    """Whole-job throughput: every rank runs the same problem `steps` times."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


def dist_barrier(dist):
    if dist is not None:
        dist.barrier()


def time_transpose(G, device, flush_buf, read_buf, peaks, n=1024, steps=50):
    """y = x^T for a 1024 x 1024 fp32 matrix (the transpose page's workload)."""
    import torch
    x = torch.rand((n, n), device=device)
    y = torch.empty_like(x)
    for _ in range(5):
        G.transpose_f32(x, n, y, n, n, n)
    torch.cuda.synchronize()
    ts = []
    for i in range(steps):
        flush_l2(flush_buf, read_buf, i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        G.transpose_f32(x, n, y, n, n, n)
        e1.record()
        ts.append((e0, e1))
    torch.cuda.synchronize()
    ms = statistics.median([a.elapsed_time(b) for a, b in ts])
    gbs = 2 * n * n * 4 / (ms * 1e-3) / 1e9
    # the same without the flush: the 4 MB matrix then stays in L2, as on the page's GPU
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        G.transpose_f32(x, n, y, n, n, n)
    e1.record()
    torch.cuda.synchronize()
    hot_us = e0.elapsed_time(e1) / steps * 1e3
    return {"workload": "transpose y = x^T, fp32 1024 x 1024", "us": ms * 1e3, "hbm_gbs": gbs,
            "frac_of_hbm_roofline": gbs / peaks["hbm_gbs"], "l2": "flushed before every step",
            "us_l2_resident_back_to_back": hot_us,
            "page_context": "0.0039 ms best on an RTX 4090 (transpose page's table; other hardware)"}


MUFU_EX2_PER_CLK_SM = 32  # special-function unit: exp2 results per clock per SM on this part


def time_score_softmax(G, device, flush_buf, read_buf, peaks, sms, steps=10, heads=None):
    """Fused score + softmax statistics on the score workload (128 heads, Q, K 4096 x 64,
    N(0,1), alpha 1/8): the 4 GiB score matrix is never stored.  The bound is the exp2
    rate of the special-function units (one exp per score), derived from the unit
    count and the maximum SM clock."""
    import torch
    from dense_fp16_gemm_tn_gb300 import inputs
    w = inputs.WORKLOADS["score_qk"]
    nb = w.batch if heads is None else heads
    g = torch.Generator(device=device)
    g.manual_seed(3000)
    Q = torch.randn((nb, w.M, w.K), generator=g, device=device).half()
    K = torch.randn((nb, w.N, w.K), generator=g, device=device).half()
    m = torch.empty((nb * w.M,), dtype=torch.float32, device=device)
    l = torch.empty_like(m)

    def call():
        G.score_softmax_stats_f16(Q, w.K, w.M * w.K, K, w.K, w.N * w.K, m, l, w.M, w.N, w.K, nb, w.alpha)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ts = []
    for i in range(steps):
        flush_l2(flush_buf, read_buf, i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        ts.append((e0, e1))
    torch.cuda.synchronize()
    st = G.gemm_tn_f16_last_device_error()
    if st != G.GEMM_OK:
        raise RuntimeError(f"device error in score+softmax timing: {G.gemm_status_string(st)}")
    ms = statistics.median([a.elapsed_time(b) for a, b in ts])
    scores = nb * w.M * w.N
    try:
        max_mhz = float(subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits",
                                        "-i", str(device.index or 0)], capture_output=True, text=True,
                                       timeout=10).stdout.split()[0])
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        max_mhz = 2070.0
    exp_peak = sms * MUFU_EX2_PER_CLK_SM * max_mhz * 1e6  # exp2 per second
    achieved = scores / (ms * 1e-3)
    return {"workload": f"fused score + scale + online softmax statistics, {nb} heads, Q,K [4096,64] N(0,1), "
                        "alpha=1/8; outputs row max and row sum (fp32)",
            "ms": ms, "tflops": w.flops * nb / w.batch / (ms * 1e-3) / 1e12,
            "scores_per_s": achieved,
            "roofline": {"bound": "alu", "achieved": achieved / 1e9, "peak": exp_peak / 1e9, "unit": "Gexp/s",
                         "frac": achieved / exp_peak,
                         "peak_source": f"{sms} SMs x {MUFU_EX2_PER_CLK_SM} exp2/clk x {max_mhz:.0f} MHz"},
            "hbm_gbs": (2 * (w.M + w.N) * w.K * nb + 8 * nb * w.M) / (ms * 1e-3) / 1e9,
            "l2": "flushed before every step"}


# Dense fp16 tensor rate per SM and clock: a 256 x 256 x 64 k-block of a CTA pair takes 512
# cycles of tcgen05.mma issue on this part (2 * 256 * 256 * 64 FLOP / 2 SMs / 512 cycles).
TENSOR_FLOP_PER_CLK_SM = 8192
HBM3E_NOMINAL_GBS = 7900.0  # the vendor's nominal HBM3e bandwidth for this part


def max_sm_mhz(device_index=0):
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits",
                              "-i", str(device_index)], capture_output=True, text=True, timeout=10).stdout
        return float(out.split()[0])
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        return 2070.0


def clock_peaks(sms, mhz):
    """Tensor peak from the SM count and the maximum SM clock (the part's own upper bound,
    what the SMs could do at full clock), with the nominal HBM3e rate."""
    return {"bf16_tflops": sms * TENSOR_FLOP_PER_CLK_SM * mhz * 1e6 / 1e12, "hbm_gbs": HBM3E_NOMINAL_GBS}


def roofline_tflops(w, peaks):
    tensor = peaks["bf16_tflops"]
    hbm = peaks["hbm_gbs"] * 1e9
    mem_bound = w.flops / (w.algorithmic_bytes / hbm) / 1e12
    return min(tensor, mem_bound), ("tensor" if tensor <= mem_bound else "hbm")


# ------------------------------------------------------------------ CPU oracle timing

def oracle_sample_seconds(w, rows, A, B, C, threads):
    """Time the oracle on the first `rows` output rows of batch entry 0 (full N and K)."""
    import numpy as np
    import oracle
    A0 = np.ascontiguousarray(A.reshape(w.batch, w.M, w.lda_)[0, :rows])
    B0 = np.ascontiguousarray(B.reshape(w.batch, w.N, w.ldb_)[0])
    C0 = np.ascontiguousarray(C.reshape(w.batch, w.M, w.ldc_)[0, :rows]) if C is not None else None
    t0 = time.perf_counter()
    oracle.gemm_tn(A0, B0, C0, rows, w.N, w.K, w.alpha, w.beta, lda=w.lda_, ldb=w.ldb_, ldc=w.ldc_, ldd=w.N,
                   threads=threads)
    return time.perf_counter() - t0


def host_inputs(w, seed):
    """Host copies (numpy uint16 bits) of the workload's operands, from the shared seeded generators."""
    from dense_fp16_gemm_tn_gb300 import inputs
    import numpy as np
    gen = inputs.uniform_half if w.dist == "uniform" else inputs.normal_half
    # Only the first batch entry is needed for a row sample.
    A = inputs.with_ld(gen(seed, w.M, w.K), w.lda_) if w.lda_ != w.K else gen(seed, w.M, w.K)
    B = inputs.with_ld(gen(seed + 1, w.N, w.K), w.ldb_) if w.ldb_ != w.K else gen(seed + 1, w.N, w.K)
    C = None
    if w.beta != 0:
        C = inputs.with_ld(gen(seed + 2, w.M, w.N), w.ldc_) if w.ldc_ != w.N else gen(seed + 2, w.M, w.N)
    w1 = type(w)(**{**w.__dict__, "batch": 1})
    return w1, np.ascontiguousarray(A), np.ascontiguousarray(B), C if C is None else np.ascontiguousarray(C)


def cpu_baseline(w, target_s=12.0):
    import oracle
    threads = oracle.default_threads()
    w1, A, B, C = host_inputs(w, 1000)
    per_row = oracle_sample_seconds(w1, 1, A, B, C, 1)  # one row, one thread: calibration
    rows = int(max(1, min(w.M, target_s * threads / max(per_row, 1e-9))))
    secs = oracle_sample_seconds(w1, rows, A, B, C, threads)
    flops = 2.0 * rows * w.N * w.K
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {rows} of {w.M} output rows of batch entry 0 (full N={w.N}, K={w.K}); "
                      f"{secs:.1f} s on {threads} host threads; fp64 accumulation"}


# ------------------------------------------------------------------ arms

def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    from dense_fp16_gemm_tn_gb300 import inputs
    oracle.build()
    w = inputs.WORKLOADS[args.workload]
    threads = oracle.default_threads()
    w1, A, B, C = host_inputs(w, 1000)
    per_row = oracle_sample_seconds(w1, 1, A, B, C, 1)
    # each step: a row sample sized so the whole run takes about 2 minutes at most
    budget_per_step = 90.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(w.M, budget_per_step * threads / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle_sample_seconds(w1, rows, A, B, C, threads)
    times = [oracle_sample_seconds(w1, rows, A, B, C, threads) for _ in range(args.steps)]
    total = sum(times)
    flops = 2.0 * rows * w.N * w.K
    value = flops * args.steps / total / 1e12
    sample = f"first {rows} of {w.M} output rows of batch entry 0 per step (full N={w.N}, K={w.K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, flushed=False),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, flushed=True):
    if not flushed:
        l2 = "n/a (CPU)"
    elif needs_flush(w):
        l2 = "flushed before every step (256 MiB write, then 256 MiB read to retire the dirty lines)"
    else:
        l2 = "operands larger than twice the 129 MB L2; not flushed"
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "batch": w.batch, "lda": w.lda_, "ldb": w.ldb_,
            "ldc": w.ldc_, "ldd": w.ldd_, "alpha": w.alpha, "beta": w.beta, "l2": l2}


def run_ours(args, rank, world, dist):
    import torch
    import dense_fp16_gemm_tn_gb300 as G
    from dense_fp16_gemm_tn_gb300 import inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    G.load_library()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    peaks, peak_src = load_peaks()
    clk_mhz = max_sm_mhz(local)
    cpeaks = clock_peaks(sms, clk_mhz)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    read_buf = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    w = inputs.WORKLOADS[args.workload]
    prob = Problem(w, device, seed=1000 + rank)
    nl, plan = launches_per_step(G, w, sms)
    with ClockSampler(local) as clk:
        times, wall = time_steps(prob, G, args.steps, args.warmup, flush, dist, read_buf)
    st = G.gemm_tn_f16_last_device_error()
    if st != G.GEMM_OK:
        raise RuntimeError(f"device error during the timed region: {G.gemm_status_string(st)}")
    total_ms = slowest_rank_ms(sum(times), dist, device)
    ms_step = total_ms / args.steps
    value = job_tflops(world, w.flops, args.steps, total_ms)

    # dominant kernel: the tensor-core GEMM; for the main workload it is the only launch of a step
    roof, bound = roofline_tflops(w, peaks)
    kernel_tflops = w.flops / (statistics.median(times) * 1e-3) / 1e12
    traffic = ncu_traffic(args.workload)
    # Steps timed back to back for half a second or more run at the part's power cap, as the
    # sustained cuBLAS loop of the measured peaks does; shorter runs compare with its burst.
    sustained = wall >= SUSTAINED_S and "bf16_tflops_sustained" in peaks
    tensor_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    tensor_src = ("bf16 cuBLAS back to back for seconds (sustained, at the power cap)" if sustained
                  else "bf16 cuBLAS burst") + "; fp16 nominal rate equals bf16"
    roofline = {"bound": "tensor" if bound == "tensor" else "hbm",
                "achieved": kernel_tflops if bound == "tensor" else w.algorithmic_bytes / (statistics.median(times) * 1e-3) / 1e9,
                "peak": tensor_peak if bound == "tensor" else peaks["hbm_gbs"],
                "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
                "traffic": traffic,
                "peak_source": f"{peak_src} ({tensor_src if bound == 'tensor' else 'STREAM copy'})"}
    if bound == "tensor":
        roofline["frac_of_burst_peak"] = kernel_tflops / peaks["bf16_tflops"]
    roofline["frac"] = roofline["achieved"] / roofline["peak"]
    if bound == "tensor":
        roofline["peak_at_max_clock"] = cpeaks["bf16_tflops"]
        roofline["frac_of_peak_at_max_clock"] = kernel_tflops / cpeaks["bf16_tflops"]
        roofline["peak_at_max_clock_source"] = (f"{sms} SMs x {TENSOR_FLOP_PER_CLK_SM} dense fp16 FLOP/clk x "
                                                f"{clk_mhz:.0f} MHz maximum SM clock")

    e2e_ms, h2d, d2h = time_e2e(prob, G, max(3, min(args.steps, 20)), 2)
    e2e = {"value": world * w.flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h}

    per_config = {}
    if not args.skip_per_config:
        for key, wk in inputs.WORKLOADS.items():
            if key == args.workload:
                continue
            pk = Problem(wk, device, seed=2000 + rank)
            steps_k = 5 if wk.flops > 1e11 else 20
            tk, _ = time_steps(pk, G, steps_k, 3, flush, dist, read_buf)
            mk = statistics.median(tk)
            rk, bk = roofline_tflops(wk, peaks)
            rn, _ = roofline_tflops(wk, cpeaks)
            tfl = wk.flops / (mk * 1e-3) / 1e12
            per_config[key] = {"workload": wk.name, "tflops": tfl, "ms": mk, "bound": bk,
                               "l2": "flushed before every step" if needs_flush(wk) else "operands exceed twice the L2; not flushed",
                               "roofline_tflops": rk, "frac_of_roofline": tfl / rk,
                               "roofline_tflops_at_max_clock": rn, "frac_of_roofline_at_max_clock": tfl / rn,
                               "frac_of_measured_peak": tfl / peaks["bf16_tflops"],
                               "hbm_gbs": wk.algorithmic_bytes / (mk * 1e-3) / 1e9}
            if wk.batch == 1:
                # end to end from page-locked host buffers through gemm_tn_f16_host
                em, eh, ed = time_e2e(pk, G, 10 if wk.flops > 1e11 else 20, 2)
                per_config[key]["e2e"] = {"value": wk.flops / (em * 1e-3) / 1e12, "unit": UNIT, "ms": em,
                                          "h2d_bytes_per_step": eh, "d2h_bytes_per_step": ed}
            if wk.flops < 1e9:
                # latency-bound: also the device time with operands left in L2 by the previous
                # call, and the cost per call of 100 calls back to back (launches pipelined)
                per_config[key]["ms_l2_hot"] = time_l2_hot(pk, G, steps_k)
                per_config[key]["ms_back_to_back"] = time_back_to_back(pk, G, 100)
            del pk
        st = G.gemm_tn_f16_last_device_error()
        if st != G.GEMM_OK:
            raise RuntimeError(f"device error in per-config timing: {G.gemm_status_string(st)}")
        per_config["transpose_f32_1024"] = time_transpose(G, device, flush, read_buf, peaks)
        per_config["score_softmax"] = time_score_softmax(G, device, flush, read_buf, peaks, sms)

    if rank != 0:
        return
    cpu = None if args.skip_cpu_baseline else cpu_baseline(w)
    clocks = clk.summary()
    if clocks.get("sm_mhz"):
        # 8192 dense fp16 FLOP per clock per SM at the SM clock sampled under load
        clocks["peak_tflops_at_sm_mhz"] = sms * 8192 * clocks["sm_mhz"] * 1e6 / 1e12
        clocks["frac_of_peak_at_sm_mhz"] = value / world / clocks["peak_tflops_at_sm_mhz"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(w),
        "frac_of_measured_peak": value / world / tensor_peak,
        "measured_peak": {"tflops": tensor_peak, "kind": "sustained" if sustained else "burst"},
        "frac_of_peak_at_max_clock": value / world / cpeaks["bf16_tflops"],
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": nl * args.steps,
        "plan": plan,
        "wall_s_timed_region": wall,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)


def run_softmax_only(args):
    import torch
    import dense_fp16_gemm_tn_gb300 as G
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(device)
    G.load_library()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    peaks, _ = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    read_buf = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    r = time_score_softmax(G, device, flush, read_buf, peaks, sms, steps=args.steps, heads=args.softmax_only)
    print(json.dumps({"score_softmax": r}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=MAIN_WORKLOAD)
    ap.add_argument("--skip-per-config", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--softmax-only", type=int, default=0, metavar="HEADS",
                    help="time only the fused score + softmax call on HEADS heads and print its entry "
                         "(a small case for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.softmax_only:
        run_softmax_only(args)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as td
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        td.init_process_group("nccl")
        dist = td
    try:
        run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
