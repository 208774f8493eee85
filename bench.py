#!/usr/bin/env python3
"""Benchmark of the GB300 weight-quantized linear layers (one JSON line on stdout, rank 0).

Default workload: decode-shaped AWQ W4A16 GEMM on the Llama-2-7B q_proj shape (K = N = 4096,
group 128, 0.1% x10 weight outliers), M in {1, 4, 16} tokens.  One step runs every M over a stack
of distinct packed copies of the layer whose total size is more than 3x the L2 cache, so every
launch streams its weights from HBM.  The step is captured once in a CUDA graph and replayed.

  value      algorithmic bytes of the step / device time (GB/s), all ranks summed
  e2e        the same, through the public call, one CUDA graph per step that copies the step's
             activations in from pinned host memory and its result (the last layer's output per M)
             back, with the host waiting for the result after every step (host clock)
  roofline   the decode kernel against the measured HBM copy bandwidth
  cpu_baseline  the CPU oracle on a bounded sample, rank 0 only

``--impl reference`` times the CPU oracle itself on the same metric (the source pages ship no
runnable code; the oracle is the reference arm).  ``--sweep FILE`` additionally measures every
hot-path row over the five workload families and writes one JSON line per case to FILE.
``--profile-case OP:DIMS`` only runs a few calls of one operation (for ncu captures).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16/W8A8 GEMM TFLOP/s & GB/s vs GB300 roofline, Llama-7B shapes, M=1..8192"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
DECODE_K, DECODE_N, DECODE_G = 4096, 4096, 128
DECODE_MS = (1, 4, 16)


# ------------------------------------------------------------------------------------------------
# algorithmic work
# ------------------------------------------------------------------------------------------------

def w4a16_bytes(M, K, N, G):
    return K * N // 2 + (K // G) * N * 2 + (K // G) * N // 2 + 2 * M * K + 2 * M * N


def w8a8_bytes(M, K, N):
    return N * K + 4 * N + M * K + 4 * M + 2 * M * N


def qrmsnorm_bytes(M, K):
    return 2 * M * K + 2 * K + M * K + 4 * M


def add_qrmsnorm_bytes(M, K):
    # x and the residual in, the new residual h out, then the QRMSNorm of h
    return 2 * M * K + 2 * M * K + 2 * M * K + 2 * K + M * K + 4 * M


def gemm_flops(M, K, N):
    return 2 * M * K * N


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        window = [r for r in rows if self.t0 is not None and self.t1 is not None and self.t0 - 0.15 <= r[0] <= self.t1 + 0.15]
        use = window if window else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {
            "sm_mhz": statistics.median([r[1] for r in use]) if use else None,
            "sm_max_mhz": max([r[2] for r in use]) if use else None,
            "reasons": reasons,
            "samples": len(window),
            "samples_total": len(rows),
        }


# ------------------------------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ------------------------------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def aggregate(local_units: float, local_seconds: float, device=None):
    """Whole-job throughput: units summed over ranks / slowest rank's time (max over ranks)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_units, local_seconds
    t = torch.tensor([local_units, local_seconds], dtype=torch.float64, device=device)
    units = t[:1].clone()
    secs = t[1:].clone()
    dist.all_reduce(units, op=dist.ReduceOp.SUM)
    dist.all_reduce(secs, op=dist.ReduceOp.MAX)
    return float(units.item()), float(secs.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------------------------------------
# ncu-derived DRAM traffic (null unless the profile was taken on the current kernel source)
# ------------------------------------------------------------------------------------------------

def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_md, src_files):
    path = os.path.join(ROOT, "profiles", profile_md)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+source_sha:\s*([0-9a-f]+)", text)
    if not m or m.group(2) != kernel_source_sha(src_files):
        return None
    return float(m.group(1))


DECODE_SRC = ["weight_quantized_linear_gb300/csrc/w4a16_decode.cu", "weight_quantized_linear_gb300/csrc/common.cuh"]


# ------------------------------------------------------------------------------------------------
# the CPU oracle as a baseline
# ------------------------------------------------------------------------------------------------

def oracle_decode_sample(target_seconds: float):
    """Time the oracle on the decode workload (one q_proj layer, every M) until ~target_seconds."""
    import numpy as np
    import oracle
    from weight_quantized_linear_gb300 import inputs
    W = inputs.weight(DECODE_K, DECODE_N, seed=0, outliers=True)
    qw, s, qz = oracle.awq_quantize(W, DECODE_G)
    xs = {m: inputs.activations(m, DECODE_K, seed=0) for m in DECODE_MS}
    done_bytes = 0
    passes = 0
    t0 = time.perf_counter()
    while True:
        for m in DECODE_MS:
            oracle.w4a16_linear(xs[m], qw, s, qz, DECODE_G)
            done_bytes += w4a16_bytes(m, DECODE_K, DECODE_N, DECODE_G)
        passes += 1
        el = time.perf_counter() - t0
        if el >= target_seconds:
            break
    return done_bytes, el, passes, oracle.num_threads()


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        oracle_decode_sample(0.0)
    t_total = 0.0
    b_total = 0
    passes = 0
    for _ in range(args.steps):
        b, el, p, cores = oracle_decode_sample(0.0)
        t_total += el
        b_total += b
        passes += p
    value = b_total / t_total / 1e9
    cores = oracle.num_threads()
    sample = (f"one step = one pass of the oracle over the q_proj layer (K=N=4096, G=128) at M=1,4,16 "
              f"(fp64 accumulation, {cores} OpenMP threads); {passes} passes timed")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": "decode W4A16 q_proj K=N=4096 G=128, M in {1,4,16}",
                                        "where": "host CPU cores"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

def l2_bytes(torch, dev):
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        return 132 * 1024 * 1024


def build_decode_workload(torch, wql, dev, layers):
    import numpy as np
    from weight_quantized_linear_gb300 import inputs
    W = torch.from_numpy(inputs.weight(DECODE_K, DECODE_N, seed=0, outliers=True)).to(dev)
    qw, s, qz = wql.awq_pack(W, DECODE_G)
    del W
    stack = [(qw, s, qz)] + [(qw.clone(), s.clone(), qz.clone()) for _ in range(layers - 1)]
    xs = {m: torch.from_numpy(inputs.activations(m, DECODE_K, seed=0)).to(dev) for m in DECODE_MS}
    ys = {m: [torch.empty((m, DECODE_N), dtype=torch.float16, device=dev) for _ in range(layers)] for m in DECODE_MS}
    return stack, xs, ys


def run_decode_step(wql, stack, xs, ys, ms=DECODE_MS):
    for m in ms:
        x = xs[m]
        for i, (qw, s, qz) in enumerate(stack):
            wql.w4a16_gemm(x, qw, s, qz, DECODE_G, out=ys[m][i])


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm the launch path outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def time_replays(torch, graph, n, stream):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            graph.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


def metric_cases(torch, wql, dev, stream, hbm, bf16, l2):
    """The rest of the metric, timed after the headline step on the same GPU: the W4A16 prefill cells
    (M in {512, 2048, 8192} x N in {4096, 11008}, K = 4096, G = 128, 1% x20 activation channels), the
    Llama-7B layer sweep at G = 128 (fused QKV 4096x12288, gate_up 4096x22016, down 11008x4096;
    M in {1, 8, 32, 128, 256}) and the SmoothQuant W8A8 block (K = 4096, N in {4096, 11008},
    M in {1, 16, 512, 4096}: the int8 GEMM alone and QRMSNorm + GEMM).  Each case is a CUDA graph of
    calls over enough distinct weight copies to exceed 3x L2; the per-call time is reported against
    the roofline that bounds it (the larger of the HBM time of its algorithmic bytes and the tensor
    time of its flops at the measured bf16 peak; int8 runs as exact fp16 on the tensor cores)."""
    import numpy as np
    from weight_quantized_linear_gb300 import inputs

    def timed(fn, copies, reps):
        g = capture(torch, fn, stream)
        g.replay()
        torch.cuda.synchronize()
        t = time_replays(torch, g, reps, stream)
        del g
        return t / (reps * copies)

    def record(cfg, op, M, K, N, G, sec, nbytes, flops, extra=None):
        t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (bf16 * 1e12)
        bound = "tensor" if t_tc > t_hbm else "hbm"
        gbs, tfs = nbytes / sec / 1e9, flops / sec / 1e12
        rec = {"config": cfg, "op": op, "M": M, "K": K, "N": N, "us": round(sec * 1e6, 3), "GB_s": round(gbs, 1),
               "TFLOP_s": round(tfs, 2), "bound": bound, "frac": round(gbs / hbm if bound == "hbm" else tfs / bf16, 4)}
        if G:
            rec["G"] = G
        if extra:
            rec.update(extra)
        return rec

    cases = []
    G = 128
    # W4A16: prefill cells and the layer sweep at G = 128
    w4 = [("prefill", M, 4096, N, False, True) for M in (512, 2048, 8192) for N in (4096, 11008)]
    w4 += [("layer sweep", M, K, N, True, False) for (K, N) in ((4096, 12288), (4096, 22016), (11008, 4096))
           for M in (1, 8, 32, 128, 256)]
    packed = {}
    for cfg, M, K, N, w_out, x_out in w4:
        key = (K, N, w_out)
        if key not in packed:
            packed.clear()
            W = torch.from_numpy(inputs.weight(K, N, seed=0, outliers=w_out)).to(dev)
            qw, sc, qz = wql.awq_pack(W, G)
            del W
            copies = int(max(2, min(64, -(-3 * l2 // w4a16_bytes(0, K, N, G)))))
            packed[key] = [(qw, sc, qz)] + [(qw.clone(), sc.clone(), qz.clone()) for _ in range(copies - 1)]
        stack = packed[key]
        x = torch.from_numpy(inputs.activations(M, K, seed=0, outlier_channels=x_out)).to(dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)

        def fn(stack=stack, x=x, y=y):
            for (a, b, z) in stack:
                wql.w4a16_gemm(x, a, b, z, G, out=y)

        flops = gemm_flops(M, K, N)
        sec = timed(fn, len(stack), 20 if flops * len(stack) < 5e12 else 3)
        kern = "tcgen05" if wql.w4a16_kernel_for(M, K, N, G) == "prefill" else "decode"
        cases.append(record(cfg, "w4a16_gemm", M, K, N, G, sec, w4a16_bytes(M, K, N, G), flops, {"kernel": kern}))
        del x, y
    packed.clear()
    # W8A8 SmoothQuant block: smoothing and quantisation on the GPU, then the GEMM and the block
    K = 4096
    for N in (4096, 11008):
        W = torch.from_numpy(inputs.weight(K, N, seed=0)).to(dev)
        copies = int(max(2, min(64, -(-3 * l2 // (N * K)))))
        for M in (1, 16, 512, 4096):
            X = torch.from_numpy(inputs.activations(M, K, seed=0, outlier_channels=True)).to(dev)
            g = torch.from_numpy(inputs.gamma(K, seed=0)).to(dev)
            a = wql.act_absmax(X, g, inputs.EPS)
            _, g2, W2 = wql.smooth(a, g, W)
            qW, ws = wql.per_channel_quant_i8(W2)
            q, xs = wql.qrmsnorm_quant_i8(X, g2, inputs.EPS)
            stack = [qW] + [qW.clone() for _ in range(copies - 1)]
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            wsp = torch.empty((max(1, wql.w8a8_workspace_bytes(M, K, N)),), dtype=torch.uint8, device=dev)

            def gemm(stack=stack, q=q, xs=xs, ws=ws, y=y, wsp=wsp):
                for w in stack:
                    wql.w8a8_gemm(q, xs, w, ws, out=y, workspace=wsp)

            def block(stack=stack, X=X, g2=g2, q=q, xs=xs, ws=ws, y=y, wsp=wsp):
                for w in stack:
                    wql.qrmsnorm_quant_i8(X, g2, inputs.EPS, q=q, xs=xs)
                    wql.w8a8_gemm(q, xs, w, ws, out=y, workspace=wsp)

            flops = gemm_flops(M, K, N)
            reps = 20 if flops * copies < 5e12 else 3
            note = {"tensor_peak_note": "exact int8 on fp16 tcgen05 (kind::i8 is absent on sm_103a); peak = measured bf16"}
            cases.append(record("w8a8 block", "w8a8_gemm", M, K, N, 0, timed(gemm, copies, reps),
                                w8a8_bytes(M, K, N), flops, note if M > 16 else None))
            cases.append(record("w8a8 block", "qrmsnorm_quant_i8+w8a8_gemm", M, K, N, 0, timed(block, copies, reps),
                                qrmsnorm_bytes(M, K) + w8a8_bytes(M, K, N), flops, note if M > 16 else None))
            del stack, y, wsp, q, xs, qW, ws, X, g, a, g2, W2
        del W
    return cases


def run_gpu(args):
    import torch
    import torch.distributed as dist
    rank, local_rank, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    from weight_quantized_linear_gb300 import build
    import weight_quantized_linear_gb300 as wql
    build.build()
    wql.load()

    hbm, bf16, bf16_sus, peak_src = peaks()
    per_layer = w4a16_bytes(0, DECODE_K, DECODE_N, DECODE_G)
    layers = max(8, -(-3 * l2_bytes(torch, dev) // per_layer) + 1)
    stack, xs, ys = build_decode_workload(torch, wql, dev, layers)
    step_bytes = sum(w4a16_bytes(m, DECODE_K, DECODE_N, DECODE_G) for m in DECODE_MS) * layers
    step_flops = sum(gemm_flops(m, DECODE_K, DECODE_N) for m in DECODE_MS) * layers
    launches_per_step = len(DECODE_MS) * layers

    stream = torch.cuda.Stream(device=dev)
    graph = capture(torch, lambda: run_decode_step(wql, stack, xs, ys), stream)
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize()
    wql.device_status(dev)

    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    # the timed region: K steps, barrier + synchronize on both sides
    barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.mark("start")
    secs = time_replays(torch, graph, args.steps, stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark("stop")
    barrier()
    # keep the GPU busy for the clock sampler when the timed region was short
    if clocks and secs < 0.5:
        extra = max(1, int(0.5 / max(secs / max(args.steps, 1), 1e-6)))
        clocks.mark("start")
        time_replays(torch, graph, extra, stream)
        clocks.mark("stop")
    clock_info = clocks.stop() if clocks else None
    wql.device_status(dev)

    units, tmax = aggregate(step_bytes * args.steps, secs, dev)
    value = units / tmax / 1e9
    ms_per_step = 1e3 * tmax / args.steps

    # per-M breakdown (device time per launch of the decode kernel)
    cases = []
    for m in DECODE_MS:
        g = capture(torch, lambda m=m: run_decode_step(wql, stack, xs, ys, ms=(m,)), stream)
        g.replay()
        torch.cuda.synchronize()
        reps = max(3, min(50, args.steps))
        t = time_replays(torch, g, reps, stream)
        per_launch = t / (reps * layers)
        b = w4a16_bytes(m, DECODE_K, DECODE_N, DECODE_G)
        cases.append({"config": "decode", "op": "w4a16_gemm", "M": m, "K": DECODE_K, "N": DECODE_N, "G": DECODE_G,
                      "us": round(per_launch * 1e6, 3), "GB_s": round(b / per_launch / 1e9, 1),
                      "TFLOP_s": round(gemm_flops(m, DECODE_K, DECODE_N) / per_launch / 1e12, 2), "bound": "hbm",
                      "frac": round(b / per_launch / 1e9 / hbm, 4), "kernel": "decode"})
        del g

    # the other configurations of the metric (prefill, layer sweep, W8A8 block), timed on this GPU
    more_cases = [] if args.no_extra_cases else metric_cases(torch, wql, dev, stream, hbm, bf16, l2_bytes(torch, dev))

    # End to end through the public call, as a serving engine replays a decode step: one CUDA graph
    # per step holds the copy of each M's activations in from pinned host memory, the 48 layers
    # (every kernel of the step) and the copy of the step's result, the last layer's output per M,
    # back to pinned host memory; the host waits for the result after every step.
    h_x = {m: xs[m].cpu().pin_memory() for m in DECODE_MS}
    h_y = {m: torch.empty((m, DECODE_N), dtype=torch.float16).pin_memory() for m in DECODE_MS}
    d_x = {m: torch.empty_like(xs[m]) for m in DECODE_MS}
    h2d = sum(h_x[m].numel() * 2 for m in DECODE_MS)
    d2h = sum(h_y[m].numel() * 2 for m in DECODE_MS)

    def e2e_body():
        for m in DECODE_MS:
            d_x[m].copy_(h_x[m], non_blocking=True)
            for i, (qw, s, qz) in enumerate(stack):
                wql.w4a16_gemm(d_x[m], qw, s, qz, DECODE_G, out=ys[m][i])
            h_y[m].copy_(ys[m][-1], non_blocking=True)

    e2e_graph = capture(torch, e2e_body, stream)

    def e2e_step():
        with torch.cuda.stream(stream):
            e2e_graph.replay()
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    barrier()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 50))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_secs = time.perf_counter() - t0
    barrier()
    e_units, e_t = aggregate(step_bytes * e2e_steps, e2e_secs, dev)
    e2e_value = e_units / e_t / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b, el, passes, cores = oracle_decode_sample(args.cpu_seconds)
        cpu = {"value": b / el / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{passes} passes of the oracle over one q_proj layer at M=1,4,16 ({el:.1f} s)"}

    achieved = step_bytes / (secs / args.steps) / 1e9
    traffic = profiled_traffic("w4a16_decode_qproj.md", DECODE_SRC)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic,
                "peak_source": f"{peak_src} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback 6.8 TB/s",
                "kernel": "w4a16_decode_kernel", "algorithmic_bytes_per_launch": round(step_bytes / launches_per_step)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": "decode W4A16 GEMM, Llama-2-7B q_proj K=N=4096, group 128, M in {1,4,16}",
                       "layers_per_step": layers, "launch": "CUDA graph, programmatic dependent launch",
                       "l2": f"inputs larger than L2: {layers} distinct packed weight copies = {layers * per_layer / 1e6:.0f} MB",
                       "parallelism": f"replicas x{world}", "tflops": round(step_flops * args.steps * world / tmax / 1e12, 3)},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "public call captured in a CUDA graph per step: pinned-host copy of x in, 48 layers x M, "
                           "last layer's y out; host waits each step"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clock_info,
            "cases": cases + more_cases,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------------------------------------
# sweep: every hot-path operation over the five workload families, one JSON line per case
# ------------------------------------------------------------------------------------------------

def run_sweep(args):
    """Times each case as a CUDA graph of calls over enough distinct weight copies that the copies
    exceed 3x L2 (or at least 2 copies); reports per-call time against the relevant roofline."""
    import numpy as np
    import torch
    from weight_quantized_linear_gb300 import build, inputs
    import weight_quantized_linear_gb300 as wql
    build.build()
    wql.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm, bf16, bf16_sus, peak_src = peaks()
    l2 = l2_bytes(torch, dev)
    stream = torch.cuda.Stream(device=dev)
    out = open(args.sweep, "w")
    wcache = {}

    def weight(K, N, outl):
        key = (K, N, outl)
        if key not in wcache:
            wcache.clear()
            wcache[key] = torch.from_numpy(inputs.weight(K, N, seed=0, outliers=outl)).to(dev)
        return wcache[key]

    def timed(fn, copies, reps):
        g = capture(torch, fn, stream)
        g.replay()
        torch.cuda.synchronize()
        t = time_replays(torch, g, reps, stream)
        del g
        return t / (reps * copies)

    rows = [r for r in (args.rows or "").split(",") if r]

    def want(*prefixes):
        """Whether any of these row families was asked for (all of them without --rows)."""
        return not rows or any(p.startswith(r) or r.startswith(p) for p in prefixes for r in rows)

    def emit(row, case, sec, nbytes, flops, bound, extra=None, peak_tensor=None):
        gbs = nbytes / sec / 1e9
        tfs = flops / sec / 1e12
        pt = bf16 if peak_tensor is None else peak_tensor
        rec = {"row": row, "case": case, "us": round(sec * 1e6, 3), "GB_s": round(gbs, 1), "TFLOP_s": round(tfs, 2),
               "bound": bound, "frac": round(gbs / hbm if bound == "hbm" else tfs / pt, 4),
               "peak": hbm if bound == "hbm" else pt, "peak_source": peak_src}
        if extra:
            rec.update(extra)
        out.write(json.dumps(rec) + "\n")
        out.flush()
        print(json.dumps(rec), flush=True)

    # a1 awq_pack (offline prep): fp32 W in, packed out
    for (K, N, G) in [(4096, 11008, 128), (4096, 22016, 32)] if want("a1") else ():
        W = weight(K, N, True)
        qw, s, qz = wql.awq_pack(W, G)
        sec = timed(lambda: wql.awq_pack(W, G), 1, 10)
        emit("a1_awq_pack", f"K{K}N{N}G{G}", sec, K * N * 4 + K * N // 2 + (K // G) * N * 2 + (K // G) * N // 2, 0, "hbm")

    # a2/a3 w4a16_gemm: tiny, decode, layer sweep, prefill
    w4 = ([("tiny", c) for c in inputs.tiny_cases()] + [("decode", c) for c in inputs.decode_cases()] +
          [("sweep", c) for c in inputs.sweep_cases()] + [("prefill", c) for c in inputs.prefill_cases()])
    packed = {}
    for fam, c in w4 if want("a2", "a3") else ():
        M, K, N, G = c["M"], c["K"], c["N"], c["G"]
        key = (K, N, G, c["w_outliers"])
        if key not in packed:
            packed.clear()
            qw, s, qz = wql.awq_pack(weight(K, N, c["w_outliers"]), G)
            per = w4a16_bytes(0, K, N, G)
            copies = int(max(2, min(64, -(-3 * l2 // per))))
            packed[key] = [(qw, s, qz)] + [(qw.clone(), s.clone(), qz.clone()) for _ in range(copies - 1)]
        stack = packed[key]
        x = torch.from_numpy(inputs.activations(M, K, seed=0, outlier_channels=c["x_outliers"])).to(dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)

        def fn(stack=stack, x=x, y=y, G=G):
            for (a, b, z) in stack:
                wql.w4a16_gemm(x, a, b, z, G, out=y)

        flops = gemm_flops(M, K, N)
        nbytes = w4a16_bytes(M, K, N, G)
        reps = 20 if flops * len(stack) < 5e12 else 3
        sec = timed(fn, len(stack), reps)
        row = "a3_w4a16_prefill" if wql.w4a16_kernel_for(M, K, N, G) == "prefill" else "a2_w4a16_decode"
        bound = "tensor" if flops / (bf16 * 1e12) > nbytes / (hbm * 1e9) else "hbm"  # the larger roofline time
        emit(row, f"{fam}:M{M}K{K}N{N}G{G}", sec, nbytes, flops, bound, {"copies": len(stack)})
        del x, y
    packed.clear()

    # a4 qrmsnorm_quant_i8 and a6 w8a8_gemm (SmoothQuant block, Llama-7B shapes); f1 its residual and
    # bias fusions; f2 the fp8 (e4m3) variant of the same block
    K = 4096
    for N in (4096, 11008) if want("a4", "a6", "f1", "f2") else ():
        W = weight(K, N, False)
        for M in (1, 16, 512, 4096):
            X = torch.from_numpy(inputs.activations(M, K, seed=0, outlier_channels=True)).to(dev)
            g = torch.from_numpy(inputs.gamma(K, seed=0)).to(dev)
            a = wql.act_absmax(X, g, inputs.EPS)
            s_, g2, W2 = wql.smooth(a, g, W)
            per = N * K
            copies = int(max(2, min(64, -(-3 * l2 // per))))
            flops = gemm_flops(M, K, N)
            reps = 20 if flops * copies < 5e12 else 3
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            R = torch.from_numpy(inputs.activations(M, K, seed=1)).to(dev)
            H = torch.empty_like(R)
            bias = torch.from_numpy(inputs.activations(1, N, seed=2)[0]).to(dev)
            RY = torch.from_numpy(inputs.activations(M, N, seed=3)).to(dev)
            if want("a4", "a6", "f1"):
                qW, ws = wql.per_channel_quant_i8(W2)
                q, xs = wql.qrmsnorm_quant_i8(X, g2, inputs.EPS)
                if N == 4096 and want("a4"):
                    # 24 calls per graph, so that graph launch overhead does not count as kernel time
                    def norms(X=X, g2=g2, q=q, xs=xs):
                        for _ in range(24):
                            wql.qrmsnorm_quant_i8(X, g2, inputs.EPS, q=q, xs=xs)

                    sec = timed(norms, 24, 20)
                    emit("a4_qrmsnorm_quant_i8", f"M{M}K{K}", sec, qrmsnorm_bytes(M, K), 0, "hbm")

                    # per_token_quant_int8 of a plain activation (no norm): 2MK in, MK + 4M out
                    def ptq(X=X, q=q, xs=xs):
                        for _ in range(24):
                            wql.per_token_quant_i8(X, q=q, xs=xs)

                    sec = timed(ptq, 24, 20)
                    emit("a4b_per_token_quant_i8", f"M{M}K{K}", sec, 3 * M * K + 4 * M, 0, "hbm")
                stack = [qW] + [qW.clone() for _ in range(copies - 1)]
                wsp = torch.empty((max(1, wql.w8a8_workspace_bytes(M, K, N)),), dtype=torch.uint8, device=dev)

                def fn8(stack=stack, q=q, xs=xs, ws=ws, y=y, wsp=wsp):
                    for w in stack:
                        wql.w8a8_gemm(q, xs, w, ws, out=y, workspace=wsp)

                sec = timed(fn8, copies, reps)
                emit("a6_w8a8_gemm", f"M{M}K{K}N{N}", sec, w8a8_bytes(M, K, N), flops, "hbm" if M <= 16 else "tensor",
                     {"copies": copies, "tensor_peak_note": "int8 run as exact fp16 on kind::f16; peak = measured bf16"})

                def block(stack=stack, X=X, g2=g2, q=q, xs=xs, ws=ws, y=y, wsp=wsp):
                    for w in stack:
                        wql.qrmsnorm_quant_i8(X, g2, inputs.EPS, q=q, xs=xs)
                        wql.w8a8_gemm(q, xs, w, ws, out=y, workspace=wsp)

                secb = timed(block, copies, reps)
                emit("a4+a6_w8a8_block", f"M{M}K{K}N{N}", secb, qrmsnorm_bytes(M, K) + w8a8_bytes(M, K, N), flops,
                     "hbm" if M <= 16 else "tensor")

                # the same block with its residual and bias fusions: h = x + r feeds the norm, and the
                # GEMM adds a bias [N] and a residual [M, N] before its single rounding to fp16
                def fused(stack=stack, X=X, R=R, H=H, g2=g2, q=q, xs=xs, ws=ws, bias=bias, RY=RY, y=y, wsp=wsp):
                    for w in stack:
                        wql.add_qrmsnorm_quant_i8(X, R, g2, inputs.EPS, residual_out=H, q=q, xs=xs)
                        wql.w8a8_gemm_fused(q, xs, w, ws, bias, RY, out=y, workspace=wsp)

                secf = timed(fused, copies, reps)
                emit("f1_w8a8_fused_block", f"M{M}K{K}N{N}", secf,
                     add_qrmsnorm_bytes(M, K) + w8a8_bytes(M, K, N) + 2 * N + 2 * M * N, flops,
                     "hbm" if M <= 16 else "tensor", {"unfused_us": round(secb * 1e6, 3)})
                del stack, wsp, q, xs, qW, ws
            if want("f2"):
                # fp8: e4m3 codes, the same byte counts as int8; the tensor roofline is the fp8 peak
                qW8, ws8 = wql.per_channel_quant_fp8(W2)
                q8, xs8 = wql.qrmsnorm_quant_fp8(X, g2, inputs.EPS)
                fp8_note = {"tensor_peak_note": "kind::f8f6f4; peak = measured bf16 x 2 (nominal fp8 / bf16 ratio)"}
                if N == 4096:
                    def norms8(X=X, g2=g2, q=q8, xs=xs8):
                        for _ in range(24):
                            wql.qrmsnorm_quant_fp8(X, g2, inputs.EPS, q=q, xs=xs)

                    sec = timed(norms8, 24, 20)
                    emit("f2_qrmsnorm_quant_fp8", f"M{M}K{K}", sec, qrmsnorm_bytes(M, K), 0, "hbm")
                stack8 = [qW8] + [qW8.clone() for _ in range(copies - 1)]

                def fnf(stack=stack8, q=q8, xs=xs8, ws=ws8, y=y):
                    for w in stack:
                        wql.w8a8_gemm_fp8(q, xs, w, ws, out=y)

                sec = timed(fnf, copies, reps)
                emit("f2_w8a8_gemm_fp8", f"M{M}K{K}N{N}", sec, w8a8_bytes(M, K, N), flops,
                     "hbm" if M <= 16 else "tensor", dict(copies=copies, **fp8_note), peak_tensor=2 * bf16)

                def fblock(stack=stack8, X=X, R=R, H=H, g2=g2, q=q8, xs=xs8, ws=ws8, bias=bias, RY=RY, y=y):
                    for w in stack:
                        wql.add_qrmsnorm_quant_fp8(X, R, g2, inputs.EPS, residual_out=H, q=q, xs=xs)
                        wql.w8a8_gemm_fp8(q, xs, w, ws, bias, RY, out=y)

                sec = timed(fblock, copies, reps)
                emit("f2_fp8_fused_block", f"M{M}K{K}N{N}", sec,
                     add_qrmsnorm_bytes(M, K) + w8a8_bytes(M, K, N) + 2 * N + 2 * M * N, flops,
                     "hbm" if M <= 16 else "tensor", fp8_note, peak_tensor=2 * bf16)
                del stack8, q8, xs8, qW8, ws8
            del y, X, a, s_, g2, W2, R, H, bias, RY

    # a5 per-channel weight quantisation (offline prep)
    if want("a5"):
        W = weight(4096, 11008, False)
        sec = timed(lambda: wql.per_channel_quant_i8(W), 1, 10)
        emit("a5_per_channel_quant_i8", "K4096N11008", sec, 4096 * 11008 * 5 + 11008 * 4, 0, "hbm")
    # f3 fused gate/up projection with SiLU(gate) * up in the epilogue (Llama-7B gate_up: K = 4096,
    # N = 2 x 11008 interleaved, G = 128), against the plain GEMM of the same weight
    if want("f3"):
        K, N, G = 4096, 22016, 128
        qw, s3, qz = wql.awq_pack(weight(K, N, True), G)
        per = w4a16_bytes(0, K, N, G)
        copies = int(max(2, min(64, -(-3 * l2 // per))))
        stack = [(qw, s3, qz)] + [(qw.clone(), s3.clone(), qz.clone()) for _ in range(copies - 1)]
        for M in (1, 8, 32, 128, 256, 2048):
            x = torch.from_numpy(inputs.activations(M, K, seed=0)).to(dev)
            y2 = torch.empty((M, N), dtype=torch.float16, device=dev)
            y1 = torch.empty((M, N // 2), dtype=torch.float16, device=dev)

            def plain(stack=stack, x=x, y=y2):
                for (a, b, z) in stack:
                    wql.w4a16_gemm(x, a, b, z, G, out=y)

            def fused(stack=stack, x=x, y=y1):
                for (a, b, z) in stack:
                    wql.w4a16_gemm_silu_mul(x, a, b, z, G, out=y)

            flops = gemm_flops(M, K, N)
            reps = 20 if flops * copies < 5e12 else 3
            tp = timed(plain, copies, reps)
            tf = timed(fused, copies, reps)
            nbytes = w4a16_bytes(M, K, N, G) - M * N  # y is [M, N / 2]
            bound = "tensor" if flops / (bf16 * 1e12) > nbytes / (hbm * 1e9) else "hbm"
            emit("f3_w4a16_gate_up_silu", f"M{M}K{K}N{N}G{G}", tf, nbytes, flops, bound,
                 {"plain_gemm_us": round(tp * 1e6, 3), "kernel": wql.w4a16_kernel_for(M, K, N, G)})
            del x, y1, y2
        del stack, qw, s3, qz

    # f4 KV cache int8 in groups of 128: Llama-7B K and V rows (2 x 32 heads x 128 channels) of
    # 16384 tokens, 256 MB of fp16, larger than L2
    if want("f4"):
        nkv, D = 16384, 8192
        kv = torch.from_numpy(inputs.activations(nkv, D, seed=4)).to(dev)
        qk, sk = wql.kv_quant_i8(kv)
        out16 = torch.empty_like(kv)
        sec = timed(lambda: wql.kv_quant_i8(kv, q=qk, scales=sk), 1, 20)
        emit("f4_kv_quant_i8", f"rows{nkv}D{D}", sec, 3 * nkv * D + 4 * nkv * (D // 128), 0, "hbm")
        sec = timed(lambda: wql.kv_dequant_i8(qk, sk, out=out16), 1, 20)
        emit("f4_kv_dequant_i8", f"rows{nkv}D{D}", sec, 3 * nkv * D + 4 * nkv * (D // 128), 0, "hbm")
        del kv, qk, sk, out16
    if want("f2"):
        W = weight(4096, 11008, False)
        sec = timed(lambda: wql.per_channel_quant_fp8(W), 1, 10)
        emit("f2_per_channel_quant_fp8", "K4096N11008", sec, 4096 * 11008 * 5 + 11008 * 4, 0, "hbm")
    wql.device_status(dev)
    out.close()
    return 0


# ------------------------------------------------------------------------------------------------
# small single-operation runs for ncu captures (no timing)
# ------------------------------------------------------------------------------------------------

def run_profile_case(args):
    """A few calls of one operation on one shape, for a profiler to capture.

    ``w4a16:M,K,N,G``, ``w8a8:M,K,N[,1]``, ``fp8:M,K,N[,1]`` (``,1``: with bias and residual),
    ``norm:M,K``, ``normfp8:M,K``, ``kv:rows,D`` (quantise then dequantise) or ``prep:K,N`` (awq_pack
    with G = 128, then per_channel_quant_i8).  Each operation is called ``--calls`` times on synthetic inputs.
    """
    import numpy as np
    import torch
    from weight_quantized_linear_gb300 import build, inputs
    import weight_quantized_linear_gb300 as wql
    build.build()
    wql.load()
    dev = torch.device("cuda", 0)
    op, _, dims = args.profile_case.partition(":")
    d = [int(v) for v in dims.split(",")] if dims else []
    calls = args.calls
    if op == "w4a16":
        M, K, N, G = d
        qw, s, qz = wql.awq_pack(torch.from_numpy(inputs.weight(K, N, seed=0, outliers=True)).to(dev), G)
        x = torch.from_numpy(inputs.activations(M, K, seed=0, outlier_channels=True)).to(dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        for _ in range(calls):
            wql.w4a16_gemm(x, qw, s, qz, G, out=y)
    elif op == "w8a8":
        M, K, N = d[:3]
        fused = len(d) > 3 and d[3] == 1  # w8a8:M,K,N,1 adds a bias and a residual in the epilogue
        rng = np.random.default_rng(0)
        q = torch.from_numpy(rng.integers(-128, 128, size=(M, K), dtype=np.int8)).to(dev)
        qW = torch.from_numpy(rng.integers(-127, 128, size=(N, K), dtype=np.int8)).to(dev)
        xs = torch.full((M,), 0.01, device=dev)
        ws = torch.full((N,), 0.001, device=dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        bias = torch.zeros((N,), dtype=torch.float16, device=dev) if fused else None
        res = torch.ones((M, N), dtype=torch.float16, device=dev) if fused else None
        for _ in range(calls):
            wql.w8a8_gemm_fused(q, xs, qW, ws, bias, res, out=y)
    elif op == "kv":
        R, D = d
        kv = torch.from_numpy(inputs.activations(R, D, seed=4)).to(dev)
        qk, sk = wql.kv_quant_i8(kv)
        out = torch.empty_like(kv)
        for _ in range(calls):
            wql.kv_quant_i8(kv, q=qk, scales=sk)
            wql.kv_dequant_i8(qk, sk, out=out)
    elif op == "fp8":
        M, K, N = d[:3]
        fused = len(d) > 3 and d[3] == 1  # fp8:M,K,N,1 adds a bias and a residual in the epilogue
        rng = np.random.default_rng(0)
        q8 = (torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)) * 60).to(wql.E4M3).to(dev)
        qW8 = (torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32)) * 60).to(wql.E4M3).to(dev)
        xs = torch.full((M,), 0.01, device=dev)
        ws = torch.full((N,), 0.001, device=dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        bias = torch.zeros((N,), dtype=torch.float16, device=dev) if fused else None
        res = torch.ones((M, N), dtype=torch.float16, device=dev) if fused else None
        for _ in range(calls):
            wql.w8a8_gemm_fp8(q8, xs, qW8, ws, bias, res, out=y)
    elif op == "normfp8":
        M, K = d
        X = torch.from_numpy(inputs.activations(M, K, seed=0, outlier_channels=True)).to(dev)
        g = torch.from_numpy(inputs.gamma(K, seed=0)).to(dev)
        for _ in range(calls):
            wql.qrmsnorm_quant_fp8(X, g, inputs.EPS)
    elif op == "norm":
        M, K = d
        X = torch.from_numpy(inputs.activations(M, K, seed=0, outlier_channels=True)).to(dev)
        g = torch.from_numpy(inputs.gamma(K, seed=0)).to(dev)
        for _ in range(calls):
            wql.qrmsnorm_quant_i8(X, g, inputs.EPS)
    elif op == "prep":
        K, N = d
        W = torch.from_numpy(inputs.weight(K, N, seed=0)).to(dev)
        for _ in range(calls):
            wql.awq_pack(W, 128)
        for _ in range(calls):
            wql.per_channel_quant_i8(W)
    else:
        raise SystemExit(f"unknown profile case {args.profile_case!r}")
    torch.cuda.synchronize()
    wql.device_status(dev)
    print("ok", flush=True)
    return 0


# Phase points stamped by the W4A16 kernels in a build with -DWQL_PHASE_TRACE (slot order).
TRACE_PHASES = {
    0: ["start", "dependency resolved", "first stage landed", "last consumer warp done", "lanes folded",
        "own slice received", "end"],
    1: ["start", "TMEM allocated", "dependency resolved", "first stage's MMAs", "last stage's MMAs",
        "last MMAs issued", "accumulator ready", "cluster barrier passed", "partials sent",
        "partials received", "outputs stored", "end", "stage 8 at the dequantisers", "stage 8 dequantised",
        "stage 8 at the MMA thread", "stage 8's MMAs issued"],
}
TRACE_END = {0: 6, 1: 11}  # the slot each CTA stamps last


def trace_summary(t, kernel):
    """Summarise phase stamps t [launches][ctas][32] (ns, 0 = not stamped) of one traced graph.

    Per phase: the median over the middle launches (the third to the second-to-last) of the median
    over a launch's CTAs, and of its earliest and latest CTA, in microseconds from the launch's
    median "dependency resolved" stamp.  Also the dependent-launch flush (this launch's dependency
    resolution after the preceding launch's last CTA end) and the launch period.
    """
    import numpy as np
    names = TRACE_PHASES[kernel]
    dep = names.index("dependency resolved")
    L = t.shape[0]
    live = t[:, :, 0] > 0
    rel = {k: [] for k in range(len(names))}
    flush, period = [], []
    prev_end = prev_dep = None
    for l in range(L):
        rows = t[l][live[l]]
        d = rows[:, dep][rows[:, dep] > 0]
        dep_t = float(np.median(d)) if d.size else float("nan")
        end_t = rows[:, TRACE_END[kernel]].max() if rows.size else 0
        if 2 <= l < L - 1:
            for k in range(len(names)):
                v = rows[:, k][rows[:, k] > 0]
                if v.size:
                    rel[k].append(((np.median(v) - dep_t) / 1e3, (v.min() - dep_t) / 1e3, (v.max() - dep_t) / 1e3))
            flush.append((dep_t - prev_end) / 1e3)
            period.append((dep_t - prev_dep) / 1e3)
        prev_end, prev_dep = end_t, dep_t
    smids = t[L // 2][live[L // 2]][:, 31]
    phases = {}
    for k, name in enumerate(names):
        if rel[k]:
            phases[name] = [round(float(np.median([r[i] for r in rel[k]])), 2) for i in range(3)]
    return {"ctas_per_launch": int(live.sum(axis=1).max()), "distinct_sms": int(np.unique(smids).size),
            "launch_period_us": round(float(np.median(period)), 2) if period else None,
            "flush_us": round(float(np.median(flush)), 2) if flush else None,
            "phases_us_from_dependency": phases}


def run_trace(args):
    """Phase trace of back-to-back W4A16 calls: ``--trace M,K,N,G``.

    Builds the developer library with the kernels' phase stamps (-DWQL_PHASE_TRACE; stamps only,
    no work skipped), runs a CUDA graph of ``--calls`` calls over distinct weight copies and output
    buffers, replays it, and prints for each phase the median over the middle launches of the
    per-launch median over CTAs, in microseconds from the launch's median "dependency resolved"
    stamp, with the spread over CTAs.  Also: the time from the preceding launch's last CTA end to
    this launch's dependency resolution (the dependent-launch flush), and the launch period.
    """
    import ctypes
    import numpy as np
    import torch
    from weight_quantized_linear_gb300 import build, inputs
    import weight_quantized_linear_gb300 as wql
    lib_path = build.build(trace=True)
    wql.load(lib_path)
    lib = wql._lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M, K, N, G = (int(v) for v in args.trace.split(","))
    kernel = int(lib.wql_w4a16_kernel_for(M, K, N, G))
    if kernel not in TRACE_PHASES:
        raise SystemExit(f"no phase trace for kernel {kernel}")
    L = max(4, args.calls)
    qw, s, qz = wql.awq_pack(torch.from_numpy(inputs.weight(K, N, seed=0, outliers=True)).to(dev), G)
    stack = [(qw, s, qz)] + [(qw.clone(), s.clone(), qz.clone()) for _ in range(L - 1)]
    x = torch.from_numpy(inputs.activations(M, K, seed=0, outlier_channels=True)).to(dev)
    ystride = (M * N * 2 + 4095) // 4096 * 4096
    yflat = torch.empty(L * ystride // 2, dtype=torch.float16, device=dev)
    ys = [yflat[l * ystride // 2: l * ystride // 2 + M * N].view(M, N) for l in range(L)]
    ctas = 2048
    buf = torch.zeros(L * ctas * 32, dtype=torch.int64, device=dev)
    st = lib.wql_trace_setup(ctypes.c_void_p(buf.data_ptr()), ctypes.c_void_p(yflat.data_ptr()), ystride, L, ctas)
    if st != 0:
        raise SystemExit(f"wql_trace_setup: {lib.wql_last_error().decode()}")
    stream = torch.cuda.Stream(device=dev)

    def fn():
        for (a, b, z), y in zip(stack, ys):
            wql.w4a16_gemm(x, a, b, z, G, out=y)
    try:
        g = capture(torch, fn, stream)
        for _ in range(3):
            g.replay()
        sec = time_replays(torch, g, 10, stream) / (10 * L)
        buf.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        wql.device_status(dev)
    finally:
        lib.wql_trace_setup(None, None, 0, 0, 0)
    t = buf.view(L, ctas, 32).cpu().numpy().astype(np.int64)
    out = {"case": f"w4a16 M={M} K={K} N={N} G={G}", "kernel": ["decode", "prefill"][kernel], "calls": L,
           "us_per_call_graph": round(sec * 1e6, 2)}
    out.update(trace_summary(t, kernel))
    print(f"{out['case']}: {out['kernel']} kernel, {out['ctas_per_launch']} CTAs on {out['distinct_sms']} SMs, "
          f"{out['us_per_call_graph']} us per call (graph of {L})")
    print(f"  preceding launch's last CTA end -> dependency resolved: {out['flush_us']:.2f} us; "
          f"period {out['launch_period_us']:.2f} us")
    print(f"  {'phase':<28} {'median':>8} {'earliest CTA':>13} {'latest CTA':>11}   (us from dependency resolved)")
    for name, (med, lo, hi) in out["phases_us_from_dependency"].items():
        print(f"  {name:<28} {med:8.2f} {lo:13.2f} {hi:11.2f}")
    print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-cases", action="store_true",
                    help="skip the prefill / layer-sweep / W8A8 cases that follow the headline timing")
    ap.add_argument("--sweep", default=None, help="measure every hot-path row; JSON lines to this file")
    ap.add_argument("--profile-case", default=None,
                    help="run one operation a few times for a profiler: w4a16:M,K,N,G | w8a8:M,K,N[,1] | fp8:M,K,N[,1] | "
                         "norm:M,K | normfp8:M,K | kv:rows,D | prep:K,N")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--trace", default=None,
                    help="phase trace of back-to-back W4A16 calls M,K,N,G (builds the -DWQL_PHASE_TRACE library; "
                         "--calls launches per graph, at least 4)")
    ap.add_argument("--rows", default=None,
                    help="with --sweep: comma-separated row families to measure (e.g. a6,f2); default all")
    args = ap.parse_args()
    if args.profile_case:
        return run_profile_case(args)
    if args.trace:
        return run_trace(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
