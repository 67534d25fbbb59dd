#!/usr/bin/env python
"""Benchmark of the quantized-matmul hot path on GB300.

Workload: the decode GEMV width sweep -- M = 1, K = N = 4096 (a 7B-class
q_proj), bits b = 1..8, group 128, zero 2^(b-1), fp16 activations and
outputs, seeded synthetic data (synthetic.decode_sweep).  One step is one
pass over the eight widths: eight qmm_gemv calls, each on its own packed
weight matrix.  The metric is the effective HBM bandwidth: algorithmic bytes
(packed weights + scales + activations + outputs, each once) per second.

Timing: the step's launches are captured once in a CUDA graph per input copy
(CPU launch overhead would otherwise dominate kernels of a few microseconds);
the inputs rotate over copies whose total exceeds twice the L2, so every step
reads its weights from HBM.  W warm-up steps, then exactly K timed steps
between a barrier + synchronize on both sides, CUDA events on the launching
stream, max over ranks.  The step consists of the eight decode-kernel launches
and nothing else, so the roofline's average launch duration is the timed step
divided by eight; per-width figures come from graphs of one width alone over
weight copies that also exceed twice the L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own replica of the sweep (weak scaling, no
collective on the data path).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Quantized-matmul effective HBM GB/s (% of ~8 TB/s roofline); TFLOP/s at M≥128"
WORKLOAD = ("decode GEMV width sweep: M=1, K=N=4096, bits 1..8, group 128, "
            "z=2^(b-1), fp16 activations/outputs, fp32 accumulation")
BITS = list(range(1, 9))
PROFILE = os.path.join(ROOT, "profiles", "qmm_gemv_decode_sweep.txt")
KERNEL_SOURCES = ["decode.cu", "decode.cuh", "decode.h", "common.cuh", "extract.cuh", "unpack_plans.h"]


def kernel_source_digest() -> str:
    """Digest of the decode kernel's sources with comments and whitespace removed,
    so that the recorded ncu traffic stays valid across comment-only edits."""
    h = hashlib.sha1()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "bit_weight_quantized_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:12]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profile_traffic():
    """ncu DRAM bytes per launch of the sweep's gemv kernels, if the committed
    capture was taken on the current kernel source; else None."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    kv = dict(line.split(":", 1) for line in text.splitlines() if ":" in line and not line.startswith(" "))
    if kv.get("kernel_source_sha1", "").strip() != kernel_source_digest():
        return None
    try:
        return float(kv["dram_bytes_per_sweep_launch_avg"].strip())
    except (KeyError, ValueError):
        return None


# ---- clocks during the timed region --------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---- distributed helpers -------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("QMM_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---- CPU oracle leg --------------------------------------------------------------------
class OracleSweep:
    """The CPU oracle on the same sweep.  Set-up (drawing the inputs, packing
    with the oracle's own packer, widening to fp64) is outside any timing; a
    step runs the oracle's dequantize-then-matmul for every width on the first
    `cols` output columns."""

    def __init__(self):
        import oracle
        import synthetic
        oracle.build()
        self.oracle = oracle
        self.probs = [synthetic.decode_sweep(b) for b in BITS]
        self.packed = [oracle.pack(p.codes, p.bits)[0] for p in self.probs]
        self.x = [p.x_f64() for p in self.probs]
        self.s = [p.scales.astype(np.float64) for p in self.probs]

    def bytes(self, cols: int) -> int:
        return sum(cols * p.K * p.bits // 8 + cols * (p.K // p.group) * 2 + p.M * p.K * 2
                   + p.M * cols * 2 for p in self.probs)

    def step(self, cols: int):
        for p, pk, x, s in zip(self.probs, self.packed, self.x, self.s):
            self.oracle.qmm(x, pk[:cols], p.bits, p.group, s[:cols], None, p.zero_const, p.K)

    def threads(self, cols: int) -> int:
        return self.oracle.threads_used(0, cols)


def oracle_baseline(sweep: OracleSweep, min_seconds: float = 3.0):
    """Whole sweep (all widths, all columns), repeated for at least min_seconds."""
    cols = sweep.probs[0].N
    sweep.step(cols)  # warm
    reps, t0 = 0, time.perf_counter()
    while True:
        sweep.step(cols)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    gbs = sweep.bytes(cols) * reps / dt / 1e9
    sample = (f"the full sweep (8 widths x 4096 columns, {sweep.bytes(cols) / 1e6:.1f} MB of "
              f"algorithmic bytes) repeated {reps} times ({dt:.1f} s)")
    return gbs, sweep.threads(cols), sample


def run_reference(args, world, rank):
    if rank != 0:
        return
    sweep = OracleSweep()
    full = sweep.probs[0].N
    # size each step so that W + K steps take about a minute
    t0 = time.perf_counter()
    sweep.step(full)
    t_full = time.perf_counter() - t0
    budget = 60.0 / max(1, args.steps + args.warmup)
    cols = int(min(full, max(16, full * budget / max(t_full, 1e-6))))
    cols = max(16, (cols // 16) * 16)
    for _ in range(args.warmup):
        sweep.step(cols)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sweep.step(cols)
    total = time.perf_counter() - t0
    value = sweep.bytes(cols) * args.steps / total / 1e9
    threads = sweep.threads(cols)
    sample = (f"every width b=1..8, first {cols} of {full} output columns, full K "
              f"(oracle fp64, {threads} threads)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)



def time_graph(torch, stream, launches, reps: int = 10, sleep: bool = True):
    """Per-launch device time (ms) of `launches` (closures) captured in one CUDA
    graph and replayed `reps` times on `stream`; inputs rotate inside `launches`."""
    with torch.cuda.stream(stream):
        for f in launches:
            f()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for f in launches:
            f()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    if sleep:
        time.sleep(0.2)   # timed as a kernel alone: the burst peak applies
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b) / (reps * len(launches))


def measure_others(torch, q, dev, stream, peak_gbs, peak_tf, gemv_kernel="auto", l2=136 << 20):
    """The other workload families, timed the same way on device-generated
    inputs of the workloads' shapes and laws (the values do not change the
    work): skinny decode (M = 16, N = 14336, b = 6, group 64), the decode
    kernel beside the skinny kernel (M = 1 and 8, K = N = 4096, b = 4), the tiled path
    (M = 128 / 512 / 2048, K = 8192, N = 28672, int4, bf16), W4A8
    (M = 1 / 16 / 64, K = N = 4096; also fed from fp16 activations through the
    per-token int8 quantizer), W8A8 (the same shapes, group 32), float6 e3m2
    weights (M = 1, K = N = 4096) and the quantizer alone (K = 4096)."""
    out = {}

    def ncopies(nbytes):
        # distinct weight copies whose total exceeds twice the L2: every launch
        # reads its weights from HBM
        return -(-2 * l2 // nbytes) + 1

    gen = torch.Generator(device=dev)
    gen.manual_seed(0)

    def codes(n, k, bits):
        return torch.randint(0, 1 << bits, (n, k), dtype=torch.uint8, device=dev, generator=gen)

    def scales(n, ng):
        return (0.02 * torch.randn(n, ng, device=dev, generator=gen).abs() + 1e-3).half()

    # skinny: M=16, N=14336, b=6, group 64, uint8 zeros
    M, N, K, b, G = 16, 14336, 4096, 6, 64
    sets = [(q.qmm_pack(codes(N, K, b), b), scales(N, K // G), codes(N, K // G, b))
            for _ in range(ncopies(N * K * b // 8))]
    x = torch.randn(M, K, device=dev, generator=gen).half()
    y = torch.empty(M, N, dtype=torch.float16, device=dev)
    ms = time_graph(torch, stream, [lambda s=s_: q.qmm_gemv(x, s[0], b, G, s[1], s[2], out=y) for s_ in sets])
    nbytes = N * K * b // 8 + N * (K // G) * 3 + M * K * 2 + M * N * 2
    out["skinny_M16_N14336_b6_g64"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                                       "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4)}
    # the same call on weights repacked to the fragment-ordered layout
    sets = [(q.qmm_repack(s[0], K, b, "tile16"), s[1], s[2]) for s in sets]
    ms = time_graph(torch, stream, [lambda s=s_: q.qmm_gemv_tile16(x, s[0], N, b, G, s[1], s[2], out=y)
                                    for s_ in sets])
    out["tile16_M16_N14336_b6_g64"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                                       "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4)}
    del sets
    # the decode kernel beside the skinny kernel (forced) on the decode shape
    # K = N = 4096, b = 4, group 128, M = 1 and 8
    N, K, b, G = 4096, 4096, 4, 128
    sets = [(q.qmm_pack(codes(N, K, b), b), scales(N, K // G)) for _ in range(ncopies(N * K * b // 8))]
    for M in (1, 8):
        x = torch.randn(M, K, device=dev, generator=gen).half()
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        nbytes = N * K * b // 8 + N * (K // G) * 2 + M * K * 2 + M * N * 2
        for kern in ("auto", "skinny"):
            q.qmm_set_gemv_kernel(kern)
            try:
                ms = time_graph(torch, stream, [lambda s=s_: q.qmm_gemv(x, s[0], b, G, s[1], None, 8, out=y)
                                                for s_ in sets])
            finally:
                q.qmm_set_gemv_kernel(gemv_kernel)
            name = "decode" if kern == "auto" else "skinny_forced"
            out[f"{name}_M{M}_N4096_b4_g128"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                                                 "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4)}
        tiled = [q.qmm_repack(s[0], K, b, "tile16") for s in sets]
        ms = time_graph(torch, stream, [lambda t=t_, s=s_: q.qmm_gemv_tile16(x, t, N, b, G, s[1], None, 8, out=y)
                                        for t_, s_ in zip(tiled, sets)])
        del tiled
        out[f"tile16_M{M}_N4096_b4_g128"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                                             "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4)}
    del sets
    # tiled: K=8192, N=28672, int4 group 128, z=8, bf16
    N, K = 28672, 8192
    wsets = [(q.qmm_pack(codes(N, K, 4), 4), scales(N, K // 128)) for _ in range(ncopies(N * K // 2))]
    for M in (128, 512, 2048):
        x = torch.randn(M, K, device=dev, generator=gen).bfloat16()
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ms = time_graph(torch, stream, [lambda w=w_: q.qmm_gemm(x, w[0], 4, 128, w[1], None, 8, out=y)
                                        for w_ in wsets], reps=3 if M == 2048 else 6)
        tf = 2.0 * M * N * K / ms / 1e9
        out[f"tiled_M{M}"] = {"us": round(ms * 1e3, 1), "TFLOPs": round(tf, 1),
                              "frac_bf16": round(tf / peak_tf, 4)}
    del wsets
    # the tiled path at the other widths: M = 512, K = 8192, N = 28672, group 128,
    # z = 2^(b-1), bf16
    M = 512
    x = torch.randn(M, K, device=dev, generator=gen).bfloat16()
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    for b in (1, 2, 3, 5, 6, 7, 8):
        wsets = [(q.qmm_pack(codes(N, K, b), b), scales(N, K // 128)) for _ in range(ncopies(N * K * b // 8))]
        ms = time_graph(torch, stream, [lambda w=w_, b=b: q.qmm_gemm(x, w[0], b, 128, w[1], None, 1 << (b - 1), out=y)
                                        for w_ in wsets], reps=3)
        tf = 2.0 * M * N * K / ms / 1e9
        out[f"tiled_M{M}_b{b}"] = {"us": round(ms * 1e3, 1), "TFLOPs": round(tf, 1),
                                   "frac_bf16": round(tf / peak_tf, 4)}
        del wsets
    # W4A8: K=N=4096, group 128
    N = K = 4096
    wsets = [(q.qmm_pack(codes(N, K, 4), 4), scales(N, K // 128)) for _ in range(ncopies(N * K // 2))]
    for M in (1, 16, 64):
        xq = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev, generator=gen)
        sa = (0.02 * torch.randn(M, device=dev, generator=gen).abs() + 1e-3).half()
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        ms = time_graph(torch, stream, [lambda w=w_: q.qmm_w4a8(xq, sa, w[0], w[1], 128, out=y) for w_ in wsets])
        nbytes = N * K // 2 + N * (K // 128) * 2 + M * K + M * 2 + M * N * 2
        out[f"w4a8_M{M}"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                             "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4),
                             "TOPs": round(2.0 * M * N * K / ms / 1e9, 1)}
        # the same from fp16 activations: per-token int8 quantizer + W4A8
        x16 = torch.randn(M, K, device=dev, generator=gen).half()
        xq_b = torch.empty(M, K, dtype=torch.int8, device=dev)
        sa_b = torch.empty(M, dtype=torch.float16, device=dev)

        def chain(w, x16=x16, xq_b=xq_b, sa_b=sa_b, y=y):
            q.qmm_quantize_act(x16, xq_b, sa_b)
            q.qmm_w4a8(xq_b, sa_b, w[0], w[1], 128, out=y)
        ms = time_graph(torch, stream, [lambda w=w_: chain(w) for w_ in wsets])
        out[f"w4a8_fp16_in_M{M}"] = {"us": round(ms * 1e3, 2), "note": "qmm_quantize_act + qmm_w4a8"}
    del wsets
    # W8A8: K = N = 4096, int8 weights, group 32 (the pages' W8A8 setting)
    wsets = [(torch.randint(-128, 128, (N, K), dtype=torch.int8, device=dev, generator=gen),
              scales(N, K // 32)) for _ in range(ncopies(N * K))]
    for M in (1, 16, 64):
        xq = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev, generator=gen)
        sa = (0.02 * torch.randn(M, device=dev, generator=gen).abs() + 1e-3).half()
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        ms = time_graph(torch, stream, [lambda w=w_: q.qmm_w8a8(xq, sa, w[0], w[1], 32, out=y) for w_ in wsets])
        nbytes = N * K + N * (K // 32) * 2 + M * K + M * 2 + M * N * 2
        out[f"w8a8_M{M}_g32"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                                 "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4),
                                 "TOPs": round(2.0 * M * N * K / ms / 1e9, 1)}
    del wsets
    # float weights on the decode kernel's tensor-core path: float6 e3m2
    # (FP6-like), M = 1, K = N = 4096, group 128
    fsets = [(q.qmm_pack(codes(N, K, 6), 6), scales(N, K // 128)) for _ in range(ncopies(N * K * 6 // 8))]
    x = torch.randn(1, K, device=dev, generator=gen).half()
    y = torch.empty(1, N, dtype=torch.float16, device=dev)
    ms = time_graph(torch, stream, [lambda w=w_: q.qmm_gemv_float(x, w[0], 3, 2, 128, w[1], out=y) for w_ in fsets])
    nbytes = N * K * 6 // 8 + N * (K // 128) * 2 + K * 2 + N * 2
    out["float6_e3m2_M1"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                             "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4)}
    del fsets
    # 4- and 8-bit float codes (e2m1, e4m3), the same shape
    for (e, m) in ((2, 1), (4, 3)):
        b = 1 + e + m
        fsets = [(q.qmm_pack(codes(N, K, b), b), scales(N, K // 128)) for _ in range(ncopies(N * K * b // 8))]
        ms = time_graph(torch, stream, [lambda w=w_, e=e, m=m: q.qmm_gemv_float(x, w[0], e, m, 128, w[1], out=y)
                                        for w_ in fsets])
        nbytes = N * K * b // 8 + N * (K // 128) * 2 + K * 2 + N * 2
        out[f"float{b}_e{e}m{m}_M1"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                                        "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4)}
    del fsets
    # per-token int8 activation quantizer alone: K = 4096, inputs rotate over 8 copies
    K = 4096
    for M in (1, 64, 2048):
        xs = [torch.randn(M, K, device=dev, generator=gen).half() for _ in range(8)]
        xq_b = torch.empty(M, K, dtype=torch.int8, device=dev)
        sa_b = torch.empty(M, dtype=torch.float16, device=dev)
        ms = time_graph(torch, stream, [lambda x=x_: q.qmm_quantize_act(x, xq_b, sa_b) for x_ in xs])
        nbytes = M * K * 2 + M * K + M * 2
        out[f"quantize_act_M{M}"] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / ms / 1e6, 1),
                                     "frac_hbm": round(nbytes / ms / 1e6 / peak_gbs, 4)}
    return out

# ---- GPU leg -------------------------------------------------------------------------------
def _libcuda():
    return ctypes.CDLL("libcuda.so.1")


def run_ours(args, world, rank, local):
    import torch
    import bit_weight_quantized_gb300 as q
    import synthetic

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q.load()
    q.qmm_set_gemv_kernel(args.gemv_kernel)
    stream = torch.cuda.Stream(device=dev)
    probs = [synthetic.decode_sweep(b) for b in BITS]
    step_bytes = sum(p.algorithmic_bytes() for p in probs)
    per_copy = sum(p.N * p.K * p.bits // 8 + p.scales.size * 2 for p in probs)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(args.copies, -(-2 * l2 // per_copy) + 1)

    # device inputs: codes packed by qmm_pack on the GPU, replicated per copy
    with torch.cuda.stream(stream):
        xs, ys, sets = [], [], []
        for p in probs:
            xs.append(torch.from_numpy(p.x.view(np.int16)).view(torch.float16).to(dev))
            ys.append(torch.empty((p.M, p.N), dtype=torch.float16, device=dev))
        base = []
        for p in probs:
            packed = q.qmm_pack(torch.from_numpy(p.codes).to(dev), p.bits)
            sc = torch.from_numpy(p.scales.view(np.int16)).view(torch.float16).to(dev)
            base.append((packed, sc))
        for c in range(copies):
            sets.append([(pk.clone(), sc.clone()) for pk, sc in base])
        stream.synchronize()

    def step(c, marks=None):
        for i, p in enumerate(probs):
            pk, sc = sets[c][i]
            if marks is not None:
                marks(2 * i)
            q.qmm_gemv(xs[i], pk, p.bits, p.group, sc, None, p.zero_const, out=ys[i])
            if marks is not None:
                marks(2 * i + 1)

    # eager warm-up (also caches device facts and kernel attributes before capture)
    with torch.cuda.stream(stream):
        for c in range(copies):
            step(c)
    stream.synchronize()
    assert q.qmm_device_status(stream) == 0

    # graph A: all copies, no events (the headline timing)
    gA = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gA, stream=stream):
        for c in range(copies):
            step(c)
    # exactly args.steps steps: whole replays of graph A, then a graph of the
    # remaining steps (copies 0 .. rem - 1)
    reps, rem = divmod(args.steps, copies)
    steps = args.steps
    gR = None
    if rem:
        gR = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gR, stream=stream):
            for c in range(rem):
                step(c)
    warm_reps = max(1, -(-args.warmup // copies))

    clocks = ClockSampler(local)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.start()
    time.sleep(0.3)
    # the warm-up steps right before the timed region (after the clock
    # sampler's start-up pause, so the timed steps do not begin on an idle GPU)
    with torch.cuda.stream(stream):
        for _ in range(warm_reps):
            gA.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            gA.replay()
        if gR is not None:
            gR.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(world, ms)
    total_bytes = sum_over_ranks(world, step_bytes * steps)
    value = total_bytes / (ms_max * 1e-3) / 1e9

    # per-width durations: for each width a graph of back-to-back launches of
    # that width alone, over distinct weight copies whose total exceeds twice
    # the L2 (HBM-cold like the headline), replayed under CUDA events on `stream`
    kdur = np.zeros(len(probs))
    for i, p in enumerate(probs):
        wb = p.N * p.K * p.bits // 8 + p.scales.size * 2
        ncp = -(-2 * l2 // wb) + 1
        wsets = [sets[c % copies][i] if c < copies else
                 (sets[0][i][0].clone(), sets[0][i][1].clone()) for c in range(ncp)]
        kdur[i] = time_graph(torch, stream,
                             [lambda w=w_, p=p, i=i: q.qmm_gemv(xs[i], w[0], p.bits, p.group, w[1], None,
                                                                p.zero_const, out=ys[i])
                              for w_ in wsets], reps=8, sleep=False)
        del wsets
    # isolated calls: each launch alone, after an L2 flush (a write of twice the
    # L2), timed by events around it; median and min of 50 per width
    flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.int32, device=dev)
    iso = {}
    with torch.cuda.stream(stream):
        for i, p in enumerate(probs):
            ts = []
            for r in range(55):
                flush.fill_(r)
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                pk, sc = sets[r % copies][i]
                a.record(stream)
                q.qmm_gemv(xs[i], pk, p.bits, p.group, sc, None, p.zero_const, out=ys[i])
                b_.record(stream)
                b_.synchronize()
                if r >= 5:
                    ts.append(a.elapsed_time(b_) * 1e3)
            iso[str(p.bits)] = (statistics.median(ts), min(ts))
    del flush
    per_width = {}
    for i, p in enumerate(probs):
        gb = p.algorithmic_bytes() / (kdur[i] * 1e-3) / 1e9
        med, mn = iso[str(p.bits)]
        per_width[str(p.bits)] = {"us": round(kdur[i] * 1e3, 3), "GBps": round(gb, 1),
                                  "isolated_us_median": round(med, 2), "isolated_us_min": round(mn, 2)}
    peak, peak_kind = measured_peaks()
    # the timed step is nothing but the eight decode-kernel launches, back to back
    # on `stream`: the kernel's average launch duration is ms_per_step / 8
    achieved = step_bytes / (ms_max / steps * 1e-3) / 1e9
    for k in per_width:
        per_width[k]["frac"] = round(per_width[k]["GBps"] / peak, 4)
    traffic = profile_traffic() if args.gemv_kernel == "auto" else None

    # e2e through the public API with host buffers: every step copies the step's
    # activations (all widths, one pinned buffer) to the device, runs the eight
    # calls, and reads all outputs back (one pinned buffer)
    xlen = [p.M * p.K for p in probs]
    ylen = [p.M * p.N for p in probs]
    xh = torch.empty(sum(xlen), dtype=torch.float16).pin_memory()
    off = 0
    for p, n in zip(probs, xlen):
        xh[off:off + n].copy_(torch.from_numpy(p.x.view(np.int16)).view(torch.float16).reshape(-1))
        off += n
    yh = torch.empty(sum(ylen), dtype=torch.float16).pin_memory()
    xd = torch.empty_like(xh, device=dev)
    yd = torch.empty_like(yh, device=dev)
    xv, yv, off_x, off_y = [], [], 0, 0
    for p, nx, ny in zip(probs, xlen, ylen):
        xv.append(xd[off_x:off_x + nx].view(p.M, p.K))
        yv.append(yd[off_y:off_y + ny].view(p.M, p.N))
        off_x += nx
        off_y += ny
    e2e_steps = max(20, min(1000, args.steps // 20))
    for it in range(e2e_steps + 5):
        if it == 5:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            c = it % copies
            xd.copy_(xh, non_blocking=True)
            for i, p in enumerate(probs):
                pk, sc = sets[c][i]
                q.qmm_gemv(xv[i], pk, p.bits, p.group, sc, None, p.zero_const, out=yv[i])
            yh.copy_(yd, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(world, e2e_s)
    e2e_value = sum_over_ranks(world, step_bytes * e2e_steps) / e2e_s / 1e9
    h2d = xh.numel() * 2
    d2h = yh.numel() * 2

    assert q.qmm_device_status(stream) == 0

    others = None
    if not args.no_others:
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                peak_tf = float(json.load(f)["bf16_tflops"])
        except Exception:
            peak_tf = 1900.0
        others = measure_others(torch, q, dev, stream, peak, peak_tf, args.gemv_kernel, l2)
        assert q.qmm_device_status(stream) == 0

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, threads, sample = oracle_baseline(OracleSweep())
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": warm_reps * copies, "ms_per_step": round(ms_max / steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "step": "8 qmm_gemv calls (b=1..8), replayed from a CUDA graph",
                       "l2": f"inputs larger than L2: {copies} rotating copies of the step's "
                             f"weights ({copies * per_copy / 1e6:.0f} MB > 2 x {l2 / 1e6:.0f} MB L2)",
                       "step_bytes": step_bytes, "parallelism": f"{world} independent replicas",
                       "gemv_kernel": args.gemv_kernel},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_kind": peak_kind,
                         "traffic": traffic,
                         "kernel": ("qmm::decode_kernel<b> (b = 1..8)" if args.gemv_kernel == "auto"
                                    else "qmm::skinny_kernel<b,1,32,0> (b = 1..8)"),
                         "algorithmic_bytes_per_launch": round(step_bytes / len(probs)),
                         "frac_of_8TBs": round(achieved / 8000.0, 4),
                         "duration_source": ("CUDA events on the launching stream around the timed "
                                             "region; the step is only the 8 decode launches (one "
                                             "per width), so the average launch takes "
                                             "ms_per_step / 8 and achieved equals value"),
                         "per_width_note": "us / GBps: one width alone, back-to-back launches over "
                                           "distinct weight copies totalling more than 2 x L2 "
                                           "(HBM-cold), CUDA events around graph replays; "
                                           "isolated_us_*: one launch after an L2 flush, events "
                                           "around it, 50 runs"},
            "per_width": per_width,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "how": "per step: one pinned host->device copy of the eight activation "
                           "vectors, eight qmm_gemv calls through the Python binding, one "
                           "device->host copy of the eight outputs, stream synchronize"},
            "gpu_launches": steps * len(probs),
            "clocks": clk,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if others is not None:
            line["others"] = others
        print(json.dumps(line), flush=True)


PROFILE_FAMILIES = ("skinny_m16", "skinny_tile16_m16", "w4a8_m64", "tiled_m128")


def run_profile_family(name: str, launches: int = 4):
    """A few eager calls of one workload family on device-generated inputs, for
    a profiler to capture one of them: the skinny batched decode (M = 16,
    N = 14336, K = 4096, b = 6, group 64, stored zeros) on the canonical or the
    fragment-ordered layout, W4A8 at M = 64 (K = N = 4096, group 128) or the tiled path at
    M = 128 (K = 8192, N = 28672, int4, bf16)."""
    import torch
    import bit_weight_quantized_gb300 as q
    q.load()
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    if name == "skinny_m16":
        M, N, K, b, G = 16, 14336, 4096, 6, 64
        pk = q.qmm_pack(torch.randint(0, 1 << b, (N, K), dtype=torch.uint8, device=dev, generator=gen), b)
        sc = (0.02 * torch.randn(N, K // G, device=dev, generator=gen).abs() + 1e-3).half()
        zz = torch.randint(0, 1 << b, (N, K // G), dtype=torch.uint8, device=dev, generator=gen)
        x = torch.randn(M, K, device=dev, generator=gen).half()
        call = lambda: q.qmm_gemv(x, pk, b, G, sc, zz)
    elif name == "skinny_tile16_m16":
        M, N, K, b, G = 16, 14336, 4096, 6, 64
        tiled = q.qmm_repack(q.qmm_pack(torch.randint(0, 1 << b, (N, K), dtype=torch.uint8, device=dev,
                                                      generator=gen), b), K, b, "tile16")
        sc = (0.02 * torch.randn(N, K // G, device=dev, generator=gen).abs() + 1e-3).half()
        zz = torch.randint(0, 1 << b, (N, K // G), dtype=torch.uint8, device=dev, generator=gen)
        x = torch.randn(M, K, device=dev, generator=gen).half()
        call = lambda: q.qmm_gemv_tile16(x, tiled, N, b, G, sc, zz)
    elif name == "w4a8_m64":
        M, N, K = 64, 4096, 4096
        w = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev, generator=gen)
        ws = (0.02 * torch.randn(N, K // 128, device=dev, generator=gen).abs() + 1e-3).half()
        xq = torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev, generator=gen)
        sa = (0.02 * torch.randn(M, device=dev, generator=gen).abs() + 1e-3).half()
        call = lambda: q.qmm_w4a8(xq, sa, w, ws, 128)
    else:
        M, N, K = 128, 28672, 8192
        w = q.qmm_pack(torch.randint(0, 16, (N, K), dtype=torch.uint8, device=dev, generator=gen), 4)
        sc = (0.02 * torch.randn(N, K // 128, device=dev, generator=gen).abs() + 1e-3).half()
        x = torch.randn(M, K, device=dev, generator=gen).bfloat16()
        call = lambda: q.qmm_gemm(x, w, 4, 128, sc, None, 8)
    for _ in range(launches):
        call()
    torch.cuda.synchronize()
    st = q.qmm_device_status()
    if st:
        raise SystemExit(f"device status {st}")
    print(json.dumps({"profile": name, "launches": launches}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--copies", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the timing of the other workload families")
    ap.add_argument("--gemv-kernel", choices=["auto", "skinny"], default="auto",
                    help="qmm_gemv's kernel: the default choice, or the skinny kernel forced "
                         "for every shape (for profiling that kernel on the sweep)")
    ap.add_argument("--profile", choices=PROFILE_FAMILIES,
                    help="run four eager calls of one workload family and exit (for a profiler)")
    args = ap.parse_args()
    if args.profile:
        run_profile_family(args.profile)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
