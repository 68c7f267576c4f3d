#!/usr/bin/env python3
"""Benchmark: Q4_K decode GEMV on GB300.

Workload (one "step"): one decode token through the quantized GEMVs of a
Llama-7B-shaped model at ncols = 1 -- 32 layers, each with the q, k, v
projections stacked into one 12288x4096 matrix, o (4096x4096), gate and up
(11008x4096 each, one fused SwiGLU launch) and down (4096x11008, fed by the
gate/up output) -- with the q8_1 quantization of every input fused into its
GEMV: 128 launches and 3.64 GB of distinct Q4_K weights per step, far larger
than the 129 MB L2, so no flush is needed.  Weights are seeded N(0, 0.02)
fp32 quantized on the device by the library's Q4_K quantizer (bit-identical
to the CPU oracle's); activations are seeded N(0, 1) with 1 % outliers x20.
The step is captured once in a CUDA graph and replayed.

Reported: weight GB/s of the whole step (value); the roofline of the GEMV
kernel over the step's own launches (algorithmic bytes over CUDA-event time
against the measured HBM copy bandwidth); microseconds per call of the
q8_1-input GEMV at the three Llama-7B shapes; an end-to-end number through
the public API with host buffers; the CPU oracle timed on the host cores;
per-call times of every other quoted workload (Q4_0, Q6_K, the column sweeps
with both decodes, the fused gate/up, the MoE variants); and bandwidth
ceilings (device copy, torch reduction, the library's read probe).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --kernel-only SHAPE|KIND|moe|q6_K:MxK|q4_0:MxK [--ncols N] [--mma-min-cols N]   (profiler captures)
  python bench.py --trace all|NAME   (per-CTA timeline of chained launches: release, staging, tail)
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
sys.path.insert(0, ROOT)

METRIC = "Q4_K/Q6_K GEMV weight GB/s and % of GB300 HBM roofline; µs/call at ncols=1"
WORKLOAD = ("llama-7b decode step, Q4_K GEMV ncols=1, q8_1 quantization fused into each GEMV: 32 layers x "
            "(qkv 12288x4096 [q,k,v stacked]; o 4096x4096; gate+up 2x11008x4096 fused SwiGLU; down 4096x11008)")
N_LAYERS = 32
D_MODEL, D_FF = 4096, 11008
Q4_K = 12
QK_K, Q4_K_BYTES = 256, 144
# launches of one layer: (name, rows, K, matrices)
STEP = [("qkv", 3 * D_MODEL, D_MODEL, 1), ("o", D_MODEL, D_MODEL, 1), ("gate_up", D_FF, D_MODEL, 2),
        ("down", D_MODEL, D_FF, 1)]
# the seven matrices of one layer, for the CPU oracle legs (same bytes as STEP)
LAYER = [("q", D_MODEL, D_MODEL, 0), ("k", D_MODEL, D_MODEL, 0), ("v", D_MODEL, D_MODEL, 0),
         ("o", D_MODEL, D_MODEL, 1), ("gate", D_FF, D_MODEL, 2), ("up", D_FF, D_MODEL, 2),
         ("down", D_MODEL, D_FF, 3)]
SHAPES = {"4096x4096": (D_MODEL, D_MODEL), "11008x4096": (D_FF, D_MODEL), "4096x11008": (D_MODEL, D_FF)}

# column count from which the plain Q4_K GEMV decodes with mma.sync (the library's default: never)
MMA_MIN_COLS = 9

# dram__bytes_read.sum + dram__bytes_write.sum per GEMV launch from one ncu
# capture, valid only while the kernel sources hash to CSRC_SHA.
TRAFFIC = {"csrc_sha": "e6fdadc3345bb932", "bytes_per_launch": 28539232,
           "shape": "mean of the step's launch kinds qkv, o, gate+up, down"}


def row_bytes(M, K):
    return K // QK_K * Q4_K_BYTES


def q8_1_bytes_unpadded(K):
    return K // 32 * 36


def algorithmic_bytes(M, K):
    """W + q8_1 activations (unpadded) + fp32 outputs for one q8_1-input GEMV launch."""
    return M * row_bytes(M, K) + q8_1_bytes_unpadded(K) + 4 * M


def fused_bytes(M, K, nmat):
    """W (nmat matrices) + fp32 activations + fp32 outputs for one fused-input launch."""
    return nmat * M * row_bytes(M, K) + 4 * K + 4 * M


def csrc_sha():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_decode_gemv_qmv_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---- clocks ----------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


# ---- distributed helpers -----------------------------------------------------------
def dist_setup(n_gpus):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v, world, device=None):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- CPU oracle timing ----------------------------------------------------------
def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine()


_CPU_INPUTS = {}


def oracle_rate(min_seconds=2.0, rows_frac=1.0, nthreads=None, kind="fp64"):
    """Weight GB/s of a CPU GEMV on one layer's matrix mix: each distinct
    shape (a row sample of it when rows_frac < 1) is timed, then weighted by
    how often it occurs in a layer.  kind "fp64": the oracle's fp64 block
    formula; "int_f32": the oracle's integer formula in fp32 (int32 block
    sums, fp32 scaling).  Returns (GB/s, threads, sample text)."""
    import oracle
    import synthetic

    nthreads = nthreads or os.cpu_count() or 1
    count = {"4096x4096": 4, "11008x4096": 2, "4096x11008": 1}
    t_layer = 0.0
    bytes_layer = 0.0
    for si, (name, (M, K)) in enumerate(SHAPES.items()):
        Ms = max(64, int(M * rows_frac))
        if (si, M) not in _CPU_INPUTS:  # quantized once, shared by every leg
            _CPU_INPUTS[(si, M)] = (
                oracle.quantize_rows(oracle.Q4_K, synthetic.weights_f32(31 + si, M, K)),
                oracle.quantize_q8_1(synthetic.activations_f32(41 + si, 1, K, outlier_frac=0.01)))
        W_all, xq = _CPU_INPUTS[(si, M)]
        W = W_all[:Ms]
        reps, t0 = 0, time.perf_counter()
        while True:
            if kind == "fp64":
                oracle.gemv_formula_mt(oracle.Q4_K, W, Ms, K, xq, 1, nthreads)
            else:
                oracle.gemv_int_f32(oracle.Q4_K, W, Ms, K, xq, 1, nthreads)
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_seconds / 3 and reps >= 2:
                break
        per_row = el / reps / Ms
        t_layer += count[name] * M * per_row
        bytes_layer += count[name] * M * row_bytes(M, K)
    what = "fp64 block-formula" if kind == "fp64" else "fp32 integer-formula"
    sample = (f"oracle {what} GEMV on {nthreads} host thread(s); one layer's matrix mix "
              f"(row fraction {rows_frac:g} of 4096x4096, 11008x4096, 4096x11008, each repeated >= "
              f"{min_seconds / 3:.1f} s) scaled by the layer's counts 4/2/1")
    return bytes_layer / t_layer / 1e9, nthreads, sample


def cpu_baselines(seconds):
    """The CPU legs: the oracle's fp64 formula and its fp32 integer formula,
    each on all host cores and on one thread (about `seconds` of CPU work each)."""
    gbs, cores, sample = oracle_rate(min_seconds=seconds)
    one, _, _ = oracle_rate(min_seconds=seconds, rows_frac=0.25, nthreads=1)
    gi, _, sample_i = oracle_rate(min_seconds=seconds, kind="int_f32")
    gi1, _, _ = oracle_rate(min_seconds=seconds, rows_frac=0.25, nthreads=1, kind="int_f32")
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
            "one_thread_gbs": round(one, 4),
            "int_f32": {"value": round(gi, 4), "one_thread_gbs": round(gi1, 4), "sample": sample_i},
            "cpu_model": cpu_model(),
            "note": "one-thread legs on a quarter of each matrix's rows; GB/s of Q4_K weights"}


# ---- reference arm: the CPU oracle as it stands ------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import synthetic

    nthreads = os.cpu_count() or 1
    # bounded sample per step: 1/8 of the rows of one layer's seven matrices
    frac = 1.0 / 8
    mats = []
    for li, (name, M, K, _) in enumerate(LAYER):
        Ms = max(16, int(M * frac))
        W = oracle.quantize_rows(oracle.Q4_K, synthetic.weights_f32(70 + li, Ms, K))
        xq = oracle.quantize_q8_1(synthetic.activations_f32(80 + li, 1, K, outlier_frac=0.01))
        mats.append((W, Ms, K, xq))
    step_bytes = sum(W.nbytes for W, _, _, _ in mats)

    def step():
        for W, Ms, K, xq in mats:
            oracle.gemv_formula_mt(oracle.Q4_K, W, Ms, K, xq, 1, nthreads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    gbs = step_bytes / (el / args.steps) / 1e9
    sample = (f"1/8 of the rows of one layer's q,k,v,o,gate,up,down Q4_K matrices ({step_bytes} weight bytes) "
              f"per step, oracle fp64 block-formula GEMV on {nthreads} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "ncols": 1, "sample": "1/8 of each matrix's rows, one layer"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- GPU arm ------------------------------------------------------------------------
def measure_ceilings(q, torch, stream, device, reps=10):
    """Diagnostic bandwidth ceilings of this GPU, measured here with CUDA events:
    a device-to-device copy of 2 GB (cudaMemcpyAsync through torch's copy_,
    counted as read + write bytes), a read-only reduction over 4 GB (torch
    sum), and this library's read probe over the same 4 GB (the GEMV weight
    stream's 128-bit L2-only loads).  The roofline denominator stays the
    measured copy figure."""
    n = 2 << 30
    src = torch.empty(n, dtype=torch.uint8, device=device)
    dst = torch.empty(n, dtype=torch.uint8, device=device)
    big = torch.ones((4 << 30) // 4, dtype=torch.float32, device=device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    out = {}
    with torch.cuda.stream(stream):
        src.fill_(1)
        for _ in range(2):
            dst.copy_(src)
        e0.record(stream)
        for _ in range(reps):
            dst.copy_(src)
        e1.record(stream)
        stream.synchronize()
        out["d2d_copy_gbs"] = round(2 * n * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
        for _ in range(2):
            big.sum()
        e0.record(stream)
        for _ in range(reps):
            big.sum()
        e1.record(stream)
        stream.synchronize()
        out["read_reduce_gbs"] = round(big.numel() * 4 * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
        sink = torch.zeros(1, dtype=torch.int32, device=device)
        for _ in range(2):
            q.read_bandwidth_probe(big, sink, stream=stream)
        e0.record(stream)
        for _ in range(reps):
            q.read_bandwidth_probe(big, sink, stream=stream)
        e1.record(stream)
        stream.synchronize()
        out["read_probe_gbs"] = round(big.numel() * 4 * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    out["note"] = ("2 GB device copy counted read+write; 4 GB float32 sum (read-only); 4 GB read by this "
                   "library's probe kernel (128-bit L2-only loads); diagnostics timed with CUDA events")
    del src, dst, big
    torch.cuda.empty_cache()
    return out


def l2_bytes(torch, device):
    return int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or (126 << 20))


def copies_for(torch, device, nbytes, floor=4):
    """Distinct weight copies a chain rotates through so that it reads at least
    three times the L2 size before any copy comes round again."""
    need = 3 * l2_bytes(torch, device)
    return max(floor, -(-need // nbytes))


def measure_configs(q, torch, stream, device, reps, peak):
    """Per-call time of the GEMV at each workload the benchmark is quoted on.
    Each launch is chained over distinct weight copies totalling at least three
    times the L2 size (so every call streams its weights from HBM) and timed
    with CUDA events as a graph of launches; a cold single call after an L2
    flush is timed beside it as a cross-check.  Returns (summary, detail):
    summary name -> [us per call, weight GB/s, fraction of the peak]."""
    import synthetic

    l2 = l2_bytes(torch, device)
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=device)

    def chain_time(calls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            stream.synchronize()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            stream.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (reps * len(calls))

    def cold_time(call, trials=5):
        """One call after writing 2x L2 of other data, events around the call alone (median)."""
        ts = []
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(trials):
                flush_buf.fill_(1)
                e0.record(stream)
                call()
                e1.record(stream)
                stream.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    def weights(t, M, K, n, seed):
        with torch.cuda.stream(stream):
            ws = [q.quantize_weights(t, synthetic.device_normal_f32(seed + i, (M, K), 0.02, device), stream=stream)
                  for i in range(n)]
        stream.synchronize()
        return ws

    def xq_of(K, nc, seed, outl=0.0):
        x = torch.from_numpy(synthetic.activations_f32(seed, nc, K, outlier_frac=outl)).to(device)
        return q.quantize_q8_1(x, stream=stream)

    summary, detail = {}, {}
    y_flat = torch.empty(8 * 32000, dtype=torch.float32, device=device)

    def yv(nc, M):  # a contiguous [nc][M] output
        return y_flat[: nc * M].view(nc, M)

    def record(name, us, wbytes, n_copies, cold=None, **extra):
        gbs = wbytes / us / 1e3
        summary[name] = [round(us, 3), round(gbs, 1), round(gbs / peak, 4)]
        detail[name] = {"us_per_call": round(us, 3), "weight_gbs": round(gbs, 1), "weight_bytes": wbytes,
                        "distinct_weight_bytes": n_copies * wbytes, **extra}
        if cold is not None:
            detail[name]["cold_us"] = round(cold, 3)

    def plain(name, t, M, K, seed, ncols=1, outl=0.0):
        wb = M * q.row_bytes(t, K)
        n = copies_for(torch, device, wb)
        ws = weights(t, M, K, n, seed)
        xq = xq_of(K, ncols, seed + 99, outl)
        calls = [lambda W=W: q.mul_mat_vec(t, W, M, K, xq, ncols, out=yv(ncols, M), stream=stream) for W in ws]
        record(name, chain_time(calls), wb, n, cold_time(calls[0]))
        del ws
        torch.cuda.empty_cache()

    plain("q4_0 4096x4096", q.Q4_0, 4096, 4096, 3_000_000)
    plain("q6_K 32000x4096", q.Q6_K, 32000, 4096, 3_000_100)
    plain("q6_K 4096x14336", q.Q6_K, 4096, 14336, 3_000_200)
    M, K = 14336, 4096
    wb = M * q.row_bytes(q.Q4_K, K)
    n14 = max(12, copies_for(torch, device, wb))
    ws = weights(q.Q4_K, M, K, n14, 3_000_300)
    for nc in range(1, 9):
        xq = xq_of(K, nc, 3_000_400 + nc)
        calls = [lambda W=W: q.mul_mat_vec(q.Q4_K, W, M, K, xq, nc, out=yv(nc, M), stream=stream) for W in ws]
        # the default decode, then the opt-in tensor-core decode at the same column count
        us = chain_time(calls)
        cold = cold_time(calls[0]) if nc == 1 else None
        q.set_mma_min_cols(q.Q4_K, 1)
        us_mma = chain_time(calls)
        q.set_mma_min_cols(q.Q4_K, 0)
        record(f"q4_K 14336x4096 nc{nc}", us, wb, n14, cold, mma_us=round(us_mma, 3))
    # the same sweep for Q6_K (4096x14336, the down projection of an 8B-class FFN)
    M6, K6 = 4096, 14336
    wb6 = M6 * q.row_bytes(q.Q6_K, K6)
    n6 = copies_for(torch, device, wb6)
    ws6 = weights(q.Q6_K, M6, K6, n6, 3_000_450)
    for nc in range(1, 9):
        xq = xq_of(K6, nc, 3_000_460 + nc)
        calls = [lambda W=W: q.mul_mat_vec(q.Q6_K, W, M6, K6, xq, nc, out=yv(nc, M6), stream=stream) for W in ws6]
        record(f"q6_K 4096x14336 nc{nc}", chain_time(calls), wb6, n6)
    del ws6
    torch.cuda.empty_cache()
    # fused gate/up, two 14336x4096 matrices per call (pairs of the copies above)
    xq = xq_of(K, 1, 3_000_500)
    pairs = [(ws[2 * i], ws[2 * i + 1]) for i in range(n14 // 2)]
    calls = [lambda g=g, u=u: q.mul_mat_vec_gate_up_swiglu(q.Q4_K, g, u, M, K, xq, 1, out=yv(1, M), stream=stream)
             for g, u in pairs]
    record("q4_K gate+up 2x14336x4096", chain_time(calls), 2 * wb, len(pairs), cold_time(calls[0]))
    # the same with the fused epilogue's up and gate biases
    bu = torch.from_numpy(synthetic.activations_f32(3_000_510, 1, M)[0]).to(device)
    bg = torch.from_numpy(synthetic.activations_f32(3_000_511, 1, M)[0]).to(device)
    calls = [lambda g=g, u=u: q.mul_mat_vec_fused(q.Q4_K, u, M, K, xq=xq, W_gate=g, bias=bu, gate_bias=bg,
                                                  out=yv(1, M), stream=stream) for g, u in pairs]
    record("q4_K gate+up 2x14336x4096 +biases", chain_time(calls), 2 * wb, len(pairs))
    # an 8B-class FFN: gate+up 2x14336x4096 then down 4096x14336, the SwiGLU
    # output handed over as fp32 (down quantizes it while staging) or as the
    # q8_1 blocks the gate+up launch writes (qmv_mul_mat_vec_fused_q8_1)
    downs = weights(q.Q4_K, K, M, len(pairs), 3_000_520)
    wbd = K * q.row_bytes(q.Q4_K, M)
    y14 = torch.empty((1, M), dtype=torch.float32, device=device)
    yq14 = torch.empty((1, q.q8_1_bytes(M)), dtype=torch.uint8, device=device)
    y4 = torch.empty((1, K), dtype=torch.float32, device=device)
    calls = []
    for (g, u), D in zip(pairs, downs):
        calls += [lambda g=g, u=u: q.mul_mat_vec_fused(q.Q4_K, u, M, K, xq=xq, W_gate=g, out=y14, stream=stream),
                  lambda D=D: q.mul_mat_vec_f32(q.Q4_K, D, K, M, y14, out=y4, stream=stream)]
    record("q4_K ffn 14336: gate+up, down; fp32 hand-off", 2 * chain_time(calls), 2 * wb + wbd, len(pairs))
    calls = []
    for (g, u), D in zip(pairs, downs):
        calls += [lambda g=g, u=u: q.mul_mat_vec_fused_q8_1(q.Q4_K, u, M, K, xq=xq, W_gate=g, want_y=False,
                                                            out_q8_1=yq14, stream=stream),
                  lambda D=D: q.mul_mat_vec(q.Q4_K, D, K, M, yq14, 1, out=y4, stream=stream)]
    record("q4_K ffn 14336: gate+up, down; q8_1 hand-off", 2 * chain_time(calls), 2 * wb + wbd, len(pairs))
    del ws, downs
    torch.cuda.empty_cache()
    # MoE: 8 experts of 14336x4096, 4 tokens, top-2 drawn without replacement;
    # the chain rotates among distinct expert sets
    ids = synthetic.moe_ids(3_000_600, 4, 2, 8)
    n_touched = len(set(ids.reshape(-1).tolist()))
    idd = torch.from_numpy(ids).to(device)
    xq4 = xq_of(K, 4, 3_000_700)
    ym = torch.empty((4, 2, M), dtype=torch.float32, device=device)
    ysh = torch.empty((4, M), dtype=torch.float32, device=device)
    n_sets = max(2, copies_for(torch, device, n_touched * wb, floor=2))
    sets = [torch.stack(weights(q.Q4_K, M, K, 8, 3_001_000 + 10 * i)).view(8, -1) for i in range(n_sets)]
    calls = [lambda E=E: q.mul_mat_vec_id(q.Q4_K, E, 8, M, K, xq4, idd, out=ym, stream=stream) for E in sets]
    record("q4_K moe 8x14336x4096 4tok top-2", chain_time(calls), n_touched * wb, n_sets, cold_time(calls[0]),
           experts_touched=n_touched)
    # the same routing plus a shared expert (every token), one launch
    shared = [weights(q.Q4_K, M, K, 1, 3_002_000 + i)[0] for i in range(n_sets)]
    calls = [lambda E=E, S=S: q.mul_mat_vec_id_fused(q.Q4_K, E, 8, M, K, idd, xq=xq4, W_shared=S, out=ym,
                                                     out_shared=ysh, stream=stream) for E, S in zip(sets, shared)]
    record("q4_K moe +shared expert", chain_time(calls), (n_touched + 1) * wb, n_sets,
           experts_touched=n_touched + 1)
    # the gated form: experts' gate matrices beside the up ones, the shared expert gated too
    gsets = [torch.stack(weights(q.Q4_K, M, K, 8, 3_003_000 + 10 * i)).view(8, -1) for i in range(n_sets)]
    gshared = [weights(q.Q4_K, M, K, 1, 3_004_000 + i)[0] for i in range(n_sets)]
    calls = [lambda E=E, G=G, S=S, SG=SG: q.mul_mat_vec_id_fused(q.Q4_K, E, 8, M, K, idd, xq=xq4, W_gate=G,
                                                                 W_shared=S, W_shared_gate=SG, out=ym, out_shared=ysh,
                                                                 stream=stream)
             for E, G, S, SG in zip(sets, gsets, shared, gshared)]
    record("q4_K moe gate/up +shared gate/up", chain_time(calls), 2 * (n_touched + 1) * wb, n_sets,
           experts_touched=n_touched + 1)
    del sets, shared, gsets, gshared, flush_buf
    torch.cuda.empty_cache()
    return summary, detail


def run_gpu(args):
    import numpy as np
    import torch

    import synthetic

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__

    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    import quantized_decode_gemv_qmv_gb300 as q

    q.set_pdl(True)
    stream = torch.cuda.Stream(device=device)

    # ---- weights: 32 layers x (qkv, o, gate + up, down), quantized on the device -----
    weights = []
    with torch.cuda.stream(stream):
        for layer in range(N_LAYERS):
            lw = {}
            for si, (name, M, K, nmat) in enumerate(STEP):
                mats = []
                for mi in range(nmat):
                    w = synthetic.device_normal_f32(1_000_000 + 100 * layer + 10 * si + mi, (M, K), 0.02, device)
                    mats.append(q.quantize_weights(Q4_K, w, stream=stream))
                    del w
                lw[name] = mats
            weights.append(lw)
    stream.synchronize()
    weight_bytes = sum(t.numel() for lw in weights for mats in lw.values() for t in mats)

    # ---- per-step inputs: attention input, attention output, FFN input per layer ---------
    n_in = 3
    xs_host = [[synthetic.activations_f32(2_000_000 + 10 * layer + i, 1, D_MODEL, outlier_frac=0.01)[0]
                for i in range(n_in)] for layer in range(N_LAYERS)]
    x_flat_host = torch.from_numpy(np.concatenate([x for lx in xs_host for x in lx])).pin_memory()
    # outputs returned to the host: qkv, o, down per layer; the SwiGLU activation stays on the device
    out_rows = [3 * D_MODEL, D_MODEL, D_MODEL]
    yoff = np.concatenate([[0], np.cumsum(out_rows * N_LAYERS)])
    acts = [torch.empty((1, D_FF), dtype=torch.float32, device=device) for _ in range(N_LAYERS)]
    # q8_1 hand-off: gate+up writes its SwiGLU output as q8_1 blocks, which down reads
    actq = [torch.empty((1, q.q8_1_bytes(D_FF)), dtype=torch.uint8, device=device) for _ in range(N_LAYERS)]
    handoff_q8_1 = args.handoff == "q8_1"

    def io_set():
        """Device input and output buffers of one step and their per-launch views."""
        xf = x_flat_host.to(device)
        yf = torch.empty(N_LAYERS * sum(out_rows), dtype=torch.float32, device=device)
        xv = [[xf[(n_in * l + i) * D_MODEL:(n_in * l + i + 1) * D_MODEL].view(1, -1) for i in range(n_in)]
              for l in range(N_LAYERS)]
        yv = [[yf[yoff[3 * l + m]:yoff[3 * l + m + 1]].view(1, -1) for m in range(3)] for l in range(N_LAYERS)]
        return xf, yf, xv, yv

    # two buffer sets: the end-to-end loop copies one step's inputs and outputs
    # while the neighbouring step computes on the other set
    io = [io_set(), io_set()]
    x_flat, y_flat, xs, ys = io[0]

    def launch(l, name, xs=xs, ys=ys):
        W = weights[l][name]
        if name == "qkv":
            q.mul_mat_vec_f32(Q4_K, W[0], 3 * D_MODEL, D_MODEL, xs[l][0], out=ys[l][0], stream=stream)
        elif name == "o":
            q.mul_mat_vec_f32(Q4_K, W[0], D_MODEL, D_MODEL, xs[l][1], out=ys[l][1], stream=stream)
        elif name == "gate_up" and handoff_q8_1:
            q.mul_mat_vec_fused_q8_1(Q4_K, W[1], D_FF, D_MODEL, x=xs[l][2], W_gate=W[0], out_q8_1=actq[l],
                                     want_y=False, stream=stream)
        elif name == "gate_up":
            q.mul_mat_vec_gate_up_swiglu_f32(Q4_K, W[0], W[1], D_FF, D_MODEL, xs[l][2], out=acts[l], stream=stream)
        elif handoff_q8_1:
            q.mul_mat_vec(Q4_K, W[0], D_MODEL, D_FF, actq[l], 1, out=ys[l][2], stream=stream)
        else:
            q.mul_mat_vec_f32(Q4_K, W[0], D_MODEL, D_FF, acts[l], out=ys[l][2], stream=stream)

    def step_calls(xs=xs, ys=ys):
        for l in range(N_LAYERS):
            for name, _, _, _ in STEP:
                launch(l, name, xs, ys)

    launches_per_step = N_LAYERS * len(STEP)

    # warm up eagerly (loads modules, caches geometry), then capture one step
    with torch.cuda.stream(stream):
        step_calls()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_calls()
    graph_b = torch.cuda.CUDAGraph()  # the same step on the second buffer set
    with torch.cuda.graph(graph_b, stream=stream):
        step_calls(io[1][2], io[1][3])
    stream.synchronize()

    # the step's launches grouped by kind (same calls, same configuration), for the roofline
    kind_graphs = {}
    for name, M, K, nmat in STEP:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(N_LAYERS):
                launch(l, name)
        kind_graphs[name] = g
    # q8_1-input GEMV chains at the three Llama-7B shapes (the pages' per-call figure)
    xq4 = q.quantize_q8_1(xs[0][0], stream=stream)
    xq11 = q.quantize_q8_1(acts[0], stream=stream)
    # 4096x4096: every o matrix and the q, k and v slices of every stacked qkv
    # (128 distinct matrices, 1.2 GB); every chain reads far more than 3x L2
    qkv_slices = [weights[l]["qkv"][0][i * D_MODEL:(i + 1) * D_MODEL] for l in range(N_LAYERS) for i in range(3)]
    shape_w = {"4096x4096": [weights[l]["o"][0] for l in range(N_LAYERS)] + qkv_slices,
               "11008x4096": [w for l in range(N_LAYERS) for w in weights[l]["gate_up"]],
               "4096x11008": [weights[l]["down"][0] for l in range(N_LAYERS)]}
    y_shape = torch.empty((1, D_FF), dtype=torch.float32, device=device)
    shape_graphs = {}
    for shape_name, (Ms, Ks) in SHAPES.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for W in shape_w[shape_name]:
                q.mul_mat_vec(Q4_K, W, Ms, Ks, xq4 if Ks == D_MODEL else xq11, 1, out=y_shape[:, :Ms], stream=stream)
        shape_graphs[shape_name] = (g, len(shape_w[shape_name]))
    stream.synchronize()

    # ---- timed region: the step ----------------------------------------------------
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(local).__enter__()  # sampled until every GPU measurement below is done
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    step_ms = ev0.elapsed_time(ev1) / args.steps
    step_ms = max_over_ranks(step_ms, world, device)
    value = world * weight_bytes / (step_ms * 1e-3) / 1e9

    def time_graph(g, n_calls, reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            stream.synchronize()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            stream.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (reps * n_calls)

    reps = max(3, min(20, args.steps // 5 or 3))
    # ---- dominant kernel: the step's GEMV launches by kind (CUDA events on the stream) --
    kinds = {}
    tot_bytes, tot_time = 0.0, 0.0
    for name, M, K, nmat in STEP:
        us = time_graph(kind_graphs[name], N_LAYERS, reps)
        b = fused_bytes(M, K, nmat)
        kinds[name] = {"rows": M, "K": K, "matrices": nmat, "us_per_call": round(us, 3),
                       "weight_gbs": round(nmat * M * row_bytes(M, K) / us / 1e3, 1),
                       "algorithmic_gbs": round(b / us / 1e3, 1)}
        tot_bytes += b * N_LAYERS
        tot_time += us * N_LAYERS
    per_shape = {}
    for shape_name, (g, n) in shape_graphs.items():
        Ms, Ks = SHAPES[shape_name]
        us = time_graph(g, n, reps)
        per_shape[shape_name] = {"us_per_call": round(us, 3), "weight_gbs": round(Ms * row_bytes(Ms, Ks) / us / 1e3, 1),
                                 "algorithmic_gbs": round(algorithmic_bytes(Ms, Ks) / us / 1e3, 1),
                                 "launches_timed": reps * n, "input": "q8_1"}
    peak, peak_kind = measured_peaks()
    # the step's 128 launches are the kernel's launches in the timed region:
    # their algorithmic bytes over the event-timed step (the average launch
    # period there); each kind chained with itself alone is a diagnostic
    achieved = tot_bytes / (step_ms * 1e3) / 1e3  # GB/s
    achieved_by_kind = tot_bytes / tot_time / 1e3
    traffic = TRAFFIC["bytes_per_launch"] if TRAFFIC["csrc_sha"] == csrc_sha() else None

    summary = {f"step {k}": [v["us_per_call"], v["weight_gbs"], round(v["weight_gbs"] / peak, 4)]
               for k, v in kinds.items()}
    summary.update({f"q4_K {k}": [v["us_per_call"], v["weight_gbs"], round(v["weight_gbs"] / peak, 4)]
                    for k, v in per_shape.items()})
    detail = {"step_kernels": kinds, "per_shape": per_shape}
    if not args.no_configs:
        cs, cd = measure_configs(q, torch, stream, device, reps, peak)
        summary.update(cs)
        detail["configs"] = cd

    # ---- end to end: host buffers, copies inside the timed region ---------------------
    # Every step copies its inputs host->device and its outputs device->host.
    # The copies run on their own streams (one per direction), double-buffered,
    # so that a step's transfers overlap the neighbouring steps' GEMVs, as a
    # serving loop would overlap them.
    y_host = [torch.empty(y_flat.numel(), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = x_flat_host.numel() * 4
    d2h = y_host[0].numel() * 4
    graphs = [graph, graph_b]
    in_stream = torch.cuda.Stream(device=device)
    out_stream = torch.cuda.Stream(device=device)

    def e2e_loop(n):
        done = [torch.cuda.Event() for _ in range(n)]
        out_done = [torch.cuda.Event() for _ in range(n)]
        start = torch.cuda.Event()
        start.record(stream)
        in_stream.wait_event(start)
        out_stream.wait_event(start)
        for k in range(n):
            b = k % 2
            in_ready = torch.cuda.Event()
            with torch.cuda.stream(in_stream):
                if k >= 2:
                    in_stream.wait_event(done[k - 2])      # step k-2 has read this set's inputs ...
                    in_stream.wait_event(out_done[k - 2])  # ... and its outputs are on the host
                io[b][0].copy_(x_flat_host, non_blocking=True)
                in_ready.record(in_stream)
            stream.wait_event(in_ready)
            graphs[b].replay()
            done[k].record(stream)
            with torch.cuda.stream(out_stream):
                out_stream.wait_event(done[k])
                y_host[b].copy_(io[b][1], non_blocking=True)
                out_done[k].record(out_stream)
        stream.wait_event(out_done[n - 1])

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e2e_loop(max(2, args.warmup))
        stream.synchronize()
        barrier(world)
        e0.record(stream)
        e2e_loop(args.steps)
        e1.record(stream)
        stream.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    e2e = world * weight_bytes / (e2e_ms * 1e-3) / 1e9
    y_flat_host = y_host[(args.steps - 1) % 2]

    if not np.all(np.isfinite(y_flat_host.numpy())):
        raise RuntimeError("non-finite GEMV output")
    if q.device_fault() != 0:
        raise RuntimeError("device fault word set during the benchmark")

    ceilings = None if args.no_configs else measure_ceilings(q, torch, stream, device)
    clk.__exit__()
    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baselines(args.cpu_seconds)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8/fp32",
        "data": "synthetic: seeded N(0,0.02) weights quantized to Q4_K on device; N(0,1) activations, 1% outliers x20",
        "config": {"workload": WORKLOAD, "ncols": 1, "layers": N_LAYERS, "weight_bytes_per_step": weight_bytes,
                   "gemv_launches_per_step": launches_per_step, "quantize_launches_per_step": 0,
                   "l2": "no flush: 3.64 GB of distinct weights per step > 129 MB L2",
                   "execution": "CUDA graph of the step, programmatic dependent launch between kernels",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "gemv_tiles_kernel<Q4_K, ncols=1, fp32 input> (the step's 128 launches, timed as the step)",
                     "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "frac_by_kind_chains": round(achieved_by_kind / peak, 4)},
        "hbm_frac_of_measured": round(value / peak, 4),
        "summary": summary,
        "summary_fields": ["us per call", "weight GB/s", f"fraction of the {peak_kind} {peak} GB/s"],
        "ceilings": ceilings,
        "e2e": {"value": round(e2e, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5),
                "copies": "every step: its inputs host->device and its outputs device->host from/to pinned host "
                          "buffers, on one copy stream per direction, double-buffered so they overlap the "
                          "neighbouring steps' GEMVs; all inside the timed region"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    # the per-launch details (decode variants, cold single calls, copies chained)
    # on a line of their own ahead of the result line, which stays compact
    print("detail: " + json.dumps(detail), flush=True)
    print(json.dumps(line), flush=True)
    return 0


def run_kernel_only(args):
    """A few GEMV launches of one shape (for profiler captures): four distinct
    weight copies rotate so consecutive launches do not hit in L2.  A config
    shape (e.g. 4096x11008) runs the q8_1-input GEMV; a step kind (qkv, o,
    gate_up, down) runs the step's fused fp32-input launch."""
    import torch

    import synthetic
    import __graft_entry__

    __graft_entry__.build()
    import quantized_decode_gemv_qmv_gb300 as q

    torch.cuda.set_device(0)
    q.set_mma_min_cols(Q4_K, args.mma_min_cols)
    kinds = {name: (M, K, nmat) for name, M, K, nmat in STEP}
    shapes = dict(SHAPES, **{"14336x4096": (14336, 4096)})
    nc = args.ncols
    qt = Q4_K
    if args.kernel_only.startswith("q6_K:") or args.kernel_only.startswith("q4_0:"):
        # another format at a config shape, q8_1 input (e.g. q6_K:4096x14336)
        fmt, shape = args.kernel_only.split(":", 1)
        qt = q.Q6_K if fmt == "q6_K" else q.Q4_0
        M, K = (int(v) for v in shape.split("x"))
        Ws = [q.quantize_weights(qt, synthetic.device_normal_f32(7 + 2 * i, (M, K), 0.02, "cuda")) for i in range(4)]
        xq = q.quantize_q8_1(torch.from_numpy(synthetic.activations_f32(9, nc, K)).cuda())
        y = torch.empty((nc, M), dtype=torch.float32, device="cuda")
        for i in range(args.launches):
            q.mul_mat_vec(qt, Ws[i % len(Ws)], M, K, xq, nc, out=y)
        torch.cuda.synchronize()
        print(json.dumps({"kernel_only": args.kernel_only, "launches": args.launches,
                          "weight_bytes_per_launch": int(Ws[0].numel())}))
        return 0
    if args.kernel_only == "moe":
        # the configs' MoE call: 8 experts of 14336x4096, 4 tokens top-2 (the same seeded routing)
        M, K = 14336, 4096
        E = torch.stack([q.quantize_weights(Q4_K, synthetic.device_normal_f32(11 + e, (M, K), 0.02, "cuda"))
                         for e in range(8)]).view(8, -1)
        ids = torch.from_numpy(synthetic.moe_ids(3_000_600, 4, 2, 8)).cuda()
        xq = q.quantize_q8_1(torch.from_numpy(synthetic.activations_f32(13, 4, K)).cuda())
        ym = torch.empty((4, 2, M), dtype=torch.float32, device="cuda")
        for _ in range(args.launches):
            q.mul_mat_vec_id(Q4_K, E, 8, M, K, xq, ids, out=ym)
        torch.cuda.synchronize()
        print(json.dumps({"kernel_only": "moe", "launches": args.launches,
                          "experts_touched": len(set(ids.view(-1).tolist()))}))
        return 0
    if args.kernel_only in shapes:
        M, K = shapes[args.kernel_only]
        nmat = 1
    elif args.kernel_only in kinds:
        M, K, nmat = kinds[args.kernel_only]
    else:
        raise SystemExit(f"unknown shape {args.kernel_only}; choose from {list(shapes) + list(kinds)}")
    Ws = [[q.quantize_weights(Q4_K, synthetic.device_normal_f32(7 + 2 * i + m, (M, K), 0.02, "cuda"))
           for m in range(nmat)] for i in range(4)]
    x = torch.from_numpy(synthetic.activations_f32(9, nc, K, outlier_frac=0.01)).cuda()
    xq = q.quantize_q8_1(x)
    y = torch.empty((nc, M), dtype=torch.float32, device="cuda")
    for i in range(args.launches):
        W = Ws[i % len(Ws)]
        if args.kernel_only in shapes:
            q.mul_mat_vec(Q4_K, W[0], M, K, xq, nc, out=y)
        elif nmat == 2:
            q.mul_mat_vec_gate_up_swiglu_f32(Q4_K, W[0], W[1], M, K, x, out=y)
        else:
            q.mul_mat_vec_f32(Q4_K, W[0], M, K, x, out=y)
    torch.cuda.synchronize()
    print(json.dumps({"kernel_only": args.kernel_only, "launches": args.launches,
                      "weight_bytes_per_launch": int(sum(w.numel() for w in Ws[0]))}))
    return 0


def run_trace(args):
    """Timeline of chained GEMV launches (per-CTA timestamps, qmv_debug_trace):
    for each workload, a CUDA graph of N launches over distinct weight copies
    (the benchmark's chained per-call setting) is replayed with the timeline on,
    and every launch k >= 1 is measured against the one before it: the PDL
    release (previous launch's last CTA done -> first wait return), the
    activation staging (wait return -> staged, median over CTAs) and its
    parts (wait return -> first activation loads returned -> own part of the
    staging done -> all activations in shared memory), the decode tail
    (median staged -> last CTA done), the spread of CTA finish times and the
    launch period (last CTA done to last CTA done)."""
    import numpy as np
    import torch

    import synthetic
    import __graft_entry__

    __graft_entry__.build()
    import quantized_decode_gemv_qmv_gb300 as q

    torch.cuda.set_device(0)
    q.set_pdl(True)
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    work = {  # name: (type, M, K, matrices, fp32 input)
        "q4_K 4096x4096 q8_1": (q.Q4_K, 4096, 4096, 1, False),
        "q4_K 14336x4096 q8_1": (q.Q4_K, 14336, 4096, 1, False),
        "q6_K 4096x14336 q8_1": (q.Q6_K, 4096, 14336, 1, False),
        "step qkv 12288x4096 fp32": (q.Q4_K, 12288, 4096, 1, True),
        "step o 4096x4096 fp32": (q.Q4_K, 4096, 4096, 1, True),
        "step gate+up 2x11008x4096 fp32": (q.Q4_K, 11008, 4096, 2, True),
        "step down 4096x11008 fp32": (q.Q4_K, 4096, 11008, 1, True),
    }
    if args.trace != "all":
        work = {k: v for k, v in work.items() if args.trace in k}
    out = {}
    for name, (t, M, K, nmat, f32) in work.items():
        wb = nmat * M * q.row_bytes(t, K)
        n = max(16, -(-3 * (126 << 20) // wb))
        with torch.cuda.stream(s):
            Ws = [[q.quantize_weights(t, synthetic.device_normal_f32(500 + 10 * i + m, (M, K), 0.02, dev), stream=s)
                   for m in range(nmat)] for i in range(n)]
        s.synchronize()
        x = torch.from_numpy(synthetic.activations_f32(77, 1, K, outlier_frac=0.01)).to(dev)
        xq = q.quantize_q8_1(x, stream=s)
        y = torch.empty((1, M), dtype=torch.float32, device=dev)
        W_ = q.TRACE_WORDS
        buf = torch.zeros(n * q.TRACE_MAX_CTAS * W_, dtype=torch.int64, device=dev)

        def chain():
            for W in Ws:
                if nmat == 2:
                    q.mul_mat_vec_gate_up_swiglu_f32(t, W[1], W[0], M, K, x, out=y, stream=s)
                elif f32:
                    q.mul_mat_vec_f32(t, W[0], M, K, x, out=y, stream=s)
                else:
                    q.mul_mat_vec(t, W[0], M, K, xq, 1, out=y, stream=s)

        with torch.cuda.stream(s):
            chain()  # eager warm-up
        s.synchronize()
        q.debug_trace(buf, n)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            chain()
        q.debug_trace(None)
        with torch.cuda.stream(s):
            for _ in range(3):
                g.replay()
            s.synchronize()
            buf.zero_()
            g.replay()
        s.synchronize()
        T = buf.view(n, q.TRACE_MAX_CTAS, W_).cpu().numpy().astype(np.float64)
        rows = []
        for k in range(1, n):
            cur = T[k][T[k][:, 0] > 0]
            prev = T[k - 1][T[k - 1][:, 0] > 0]
            prev_done = prev[:, 5].max()
            rows.append([cur[:, 1].min() - prev_done,                # release
                         np.median(cur[:, 4] - cur[:, 1]),            # staging
                         np.median(cur[:, 2] - cur[:, 1]),            #   wait -> first loads returned
                         np.median(cur[:, 3] - cur[:, 2]),            #   first loads -> own part done
                         np.median(cur[:, 4] - cur[:, 3]),            #   own part -> all activations in
                         cur[:, 5].max() - np.median(cur[:, 4]),      # decode tail
                         cur[:, 5].max() - np.median(cur[:, 5]),      # last CTA behind the median one
                         cur[:, 0].min() - prev_done,                 # first CTA entry (negative: early)
                         cur[:, 5].max() - prev_done])                # period
        r = np.median(np.asarray(rows), axis=0) / 1e3
        # the staging parts need stamps [2] and [3], which only the coalesced
        # staging paths write (not the per-unit q8_1 staging)
        parts = bool(np.all(T[1:, :, 2][T[1:, :, 0] > 0] > 0))
        part = (lambda v: round(v, 3)) if parts else (lambda v: None)
        out[name] = {"release_us": round(r[0], 3), "staging_us": round(r[1], 3), "first_loads_us": part(r[2]),
                     "own_part_us": part(r[3]), "complete_us": part(r[4]), "tail_us": round(r[5], 3),
                     "last_cta_behind_median_us": round(r[6], 3), "first_entry_us": round(r[7], 3),
                     "period_us": round(r[8], 3), "ideal_us": round(wb / 6668.5e3, 3), "launches": n - 1,
                     "ctas": int((T[1][:, 0] > 0).sum())}
        print(json.dumps({name: out[name]}), flush=True)
        del Ws, buf
        torch.cuda.empty_cache()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=6.0, help="CPU-baseline timing budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config timing section")
    ap.add_argument("--handoff", choices=["fp32", "q8_1"], default="fp32",
                    help="how the SwiGLU output reaches the down projection in the step")
    ap.add_argument("--kernel-only", default=None,
                    help="profiling aid: only GEMV launches of one shape, step kind, or the MoE call (moe)")
    ap.add_argument("--launches", type=int, default=8)
    ap.add_argument("--ncols", type=int, default=1, help="profiling aid: activation columns of a --kernel-only shape")
    ap.add_argument("--trace", default=None,
                    help="timeline of chained launches (per-CTA timestamps): 'all' or a substring of a workload name")
    ap.add_argument("--mma-min-cols", type=int, default=0,
                    help="profiling aid: columns from which --kernel-only uses the tensor-core decode (0: default)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel_only:
        return run_kernel_only(args)
    if args.trace:
        return run_trace(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
