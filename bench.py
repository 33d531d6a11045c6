#!/usr/bin/env python3
"""Decode tokens/s of the Qwen3-8B-shaped Q4_K/Q6_K stack at M = 1 on GB300.

Default arm (ours): one decode token per step through libdq (the persistent
token kernel: one cooperative launch per token) on synthetic random-init
weights (4.65 GB, larger than L2, read once per step).  Prints one JSON line
with the metric, the roofline of the timed kernel, the end-to-end number
through the C ABI with host buffers, clock samples and the CPU-oracle
baseline; the separate-kernel CUDA graph (182 kernels) is timed beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the token does not shard across GPUs here); the time is the max over ranks.
The reference arm (--impl reference) times the fp64 CPU oracle on this host's
cores on the same workload, one token per step; rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantised_gemv_norm_gb300 import ledger, synth  # noqa: E402

METRIC = "decode tokens/s (Qwen3-8B-shaped Q4_K, M=1); achieved HBM GB/s vs GB300 peak"
SEED = 1
MAX_CTX = 1024
WORKLOAD = ("Qwen3-8B-shaped decode token: 36 layers (Q4_K attention q|k|v 6144x4096 and o 4096x4096, "
            "Q4_K gate/up 12288x4096, down 4096x12288 Q6_K in odd layers / Q4_K in even), final RMSNorm, "
            "Q6_K vocabulary 151936x4096; Qwen3 attention inputs (per-head q/k RMSNorm, rotary base 1e6); "
            "empty KV cache (pos 0); M=1")
# The pages' own number for this workload: llama.cpp, Qwen3-8B Q4_K, empty context, RTX 5090
# ("The roofline holds on a second GPU", "How I ran it": 248.8 / 253.9 / 255.1 tok/s); median.
PAGES_BASELINE_TOK_S = 253.9
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0  # dense, burst; fp16 runs at the same tensor rate
KERNEL_KINDS = ("qkv", "attention", "o_proj", "gate_up", "down", "vocab")
# The arithmetic of the timed path: 4- and 6-bit integer weight codes times the
# activation as 15-bit fixed point per 32-element group, integer dot products
# (dp2a, int32), block and group scales applied and accumulated in fp32.
DTYPE = "q4k/q6k codes x s16 group fixed-point activations, int32 dot, f32 scale+accumulate"


def bench_config(world: int) -> dict:
    """The workload both arms run (identical keys and values for the same N)."""
    return {"workload": WORKLOAD, "bytes_per_token": token_bytes(0), "ctx": 0,
            "l2": "inputs larger than L2: 4.65 GB of weights read per step, no flush needed",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def aggregate_max(value: float, world: int, device=None) -> float:
    """Max over ranks (the job's time is its slowest rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return None, "fallback"


def tensor_peak_tflops():
    d, _ = measured_peaks()
    if d:
        for key in ("bf16_tflops", "bf16_TFLOPs"):
            if key in d and isinstance(d[key], (int, float)):
                return float(d[key]), "of measured"
    return FALLBACK_BF16_TFLOPS, "of fallback"


def hbm_peak_gbs():
    d, src = measured_peaks()
    if d:
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in d and isinstance(d[key], (int, float)):
                return float(d[key]), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms while the GPU runs the
    decode steps (warm-up, timed and end-to-end regions)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), "dq_bench_clocks_%d_%d.csv" % (gpu_index, os.getpid()))

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def wait_first_sample(self, timeout_s: float = 3.0):
        t0 = time.time()
        while self.proc and time.time() - t0 < timeout_s:
            try:
                if os.path.getsize(self.path) > 0:
                    return
            except OSError:
                pass
            time.sleep(0.02)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def token_bytes(ctx: int) -> int:
    S = ledger.QWEN3_8B_SHAPE
    return ledger.token_bytes(S["n_layers"], S["hidden"], S["ffn"], S["n_q"], S["n_kv"], S["hd"], S["vocab"], ctx)


def kernel_bytes(kind: str, layer: int, ctx: int) -> int:
    """Algorithmic bytes of one launch: weights (+ gamma, + K/V read)."""
    S = ledger.QWEN3_8B_SHAPE
    H, F = S["hidden"], S["ffn"]
    qkv_rows = (S["n_q"] + 2 * S["n_kv"]) * S["hd"]
    if kind == "qkv":
        return ledger.matrix_bytes(ledger.FMT_Q4K, qkv_rows, H) + 4 * H
    if kind == "attention":
        return ledger.kv_read_bytes(1, S["n_kv"], S["hd"], ctx + 1)
    if kind == "o_proj":
        return ledger.matrix_bytes(ledger.FMT_Q4K, H, S["n_q"] * S["hd"])
    if kind == "gate_up":
        return 2 * ledger.matrix_bytes(ledger.FMT_Q4K, F, H) + 4 * H
    if kind == "down":
        fmt = ledger.FMT_Q6K if layer % 2 == 1 else ledger.FMT_Q4K
        return ledger.matrix_bytes(fmt, H, F)
    return ledger.matrix_bytes(ledger.FMT_Q6K, S["vocab"], H) + 4 * H


# ------------------------------------------------------------------ ours


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    from quantised_gemv_norm_gb300 import build, dq, upload

    build.build()
    dq.load()
    t0 = time.time()
    m = synth.make_model(SEED, max_ctx=MAX_CTX, qwen3_attention=True, **synth.QWEN3_8B)
    kv = synth.make_kv_cache(SEED, m, 0)
    w = upload.to_device(m, kv, device)
    # The token as one persistent cooperative kernel (the library's fastest mode where
    # the shape allows); the separate-kernel CUDA graph is timed beside it.
    model = dq.Model(**upload.model_kwargs(m), weights=w, use_graph=True,
                     flags=0 if args.no_fused else dq.MODEL_FUSED)
    mode = "fused token kernel" if model.fused else "CUDA graph of separate kernels"
    setup_s = time.time() - t0
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream

    K, W = args.steps, args.warmup
    xs = torch.stack([torch.from_numpy(synth.decode_input(SEED, m.hidden, t)) for t in range(K + W)]).to(device)
    logits = torch.empty(m.vocab, dtype=torch.float32, device=device)

    def timed_steps(mdl, pos):
        for t in range(W):
            mdl.step_raw(xs[t].data_ptr(), pos, logits.data_ptr(), sh)
        torch.cuda.synchronize(device)
        barrier(world, device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        a.record(stream)
        for t in range(K):
            mdl.step_raw(xs[W + t].data_ptr(), pos, logits.data_ptr(), sh)
        b.record(stream)
        torch.cuda.synchronize(device)
        barrier(world, device)
        return aggregate_max(a.elapsed_time(b) / 1e3, world, device)

    # ---- device-timed decode: inputs resident in HBM, pos 0 (empty cache) each step.
    # The clock sampler runs from before the warm-up through the end-to-end steps below
    # (nvidia-smi takes a moment to start: the first sample is awaited first).
    clocks = ClockSampler(device.index if device.index is not None else 0).__enter__()
    clocks.wait_first_sample()
    max_s = timed_steps(model, 0)
    err = dq.device_error()
    tok_s = K * world / max_s

    # ---- end to end through the C ABI with host buffers: pinned x in, logits out, per step
    x_host = torch.from_numpy(np.stack([synth.decode_input(SEED + 7, m.hidden, t) for t in range(K + W)])).pin_memory()
    out_host = torch.empty(m.vocab, dtype=torch.float32).pin_memory()

    def e2e_step(t):  # dq_decode_step_host: copy in, token, copy out, wait
        model.step_host(x_host[t], 0, out_host)

    for t in range(W):
        e2e_step(t)
    barrier(world, device)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for t in range(K):
        e2e_step(W + t)
    torch.cuda.synchronize(device)
    e2e_local = time.perf_counter() - t0
    clocks.__exit__(None, None, None)
    barrier(world, device)
    e2e_max = aggregate_max(e2e_local, world, device)

    # ---- roofline of the timed kernel: the whole token's algorithmic bytes per launch over
    # its launch time (CUDA events on the launching stream, the timed region above)
    tb = token_bytes(0)
    peak, peak_src = hbm_peak_gbs()
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        try:
            traffic = json.load(open(prof)).get("token_kernel" if model.fused else "gate_up", {}).get(
                "dram_bytes_per_launch")
        except Exception:
            traffic = None
    if model.fused:
        rl_kernel, achieved = "token_kernel", round(tb * K / max_s / 1e9, 1)
    else:
        rl_kernel, achieved = None, None

    # ---- the separate-kernel path: the CUDA graph of 182 PDL-chained kernels, and each
    # kernel kind alone (each kind across all 36 layers, CUDA events on this stream).
    # The per-kind launches are queued behind a short device-side sleep before the first
    # event, so the events time the GPU running them back to back, not the host issuing
    # them; they are chained with programmatic dependent launch as in the token.
    gmodel = dq.Model(**upload.model_kwargs(m), weights=w, use_graph=True)
    gs = timed_steps(gmodel, 0)
    per_kernel = {}
    for kind_i, kind in enumerate(KERNEL_KINDS):
        layers = [0] if kind == "vocab" else list(range(m.n_layers))
        reps = 3 if kind == "vocab" else 1
        for l in layers[:2]:
            gmodel.enqueue_kernel(l, kind_i, sh)
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(20_000_000)  # about 10 ms at 2 GHz: longer than queuing the launches takes
        a.record(stream)
        for _ in range(reps):
            for l in layers:
                gmodel.enqueue_kernel(l, kind_i, sh)
        b.record(stream)
        torch.cuda.synchronize(device)
        n = reps * len(layers)
        us = a.elapsed_time(b) * 1e3 / n
        byts = sum(kernel_bytes(kind, l, 0) for l in layers) / len(layers)
        per_kernel[kind] = {"us_per_launch": round(us, 3), "bytes_per_launch": int(byts),
                            "GBps": round(byts / us / 1e3, 1), "launches_per_token": len(layers)}
    share = {k: v["us_per_launch"] * v["launches_per_token"] for k, v in per_kernel.items()}
    dom = max(share, key=share.get)
    dom_traffic = None
    if os.path.exists(prof):
        try:
            dom_traffic = json.load(open(prof)).get(dom, {}).get("dram_bytes_per_launch")
        except Exception:
            dom_traffic = None
    separate = {"tokens_per_s": round(K * world / gs, 2), "ms_per_step": round(gs / K * 1e3, 4),
                "launches_per_step": gmodel.launches_per_step, "per_kernel": per_kernel,
                "dominant_kernel": dom, "dominant_frac": round(per_kernel[dom]["GBps"] / peak, 4),
                "dominant_traffic": dom_traffic}
    gmodel.close()
    if rl_kernel is None:  # the separate kernels are what ran: the dominant one
        rl_kernel, achieved = dom, per_kernel[dom]["GBps"]

    # ---- 512-token context (cache filled with N(0,1) fp16, pos 512)
    ctx = {}
    if not args.no_ctx512:
        kv512 = synth.make_kv_cache(SEED + 1, m, 512)
        w["kv_cache"].copy_(torch.from_numpy(kv512.view(np.int16)).to(device))
        del kv512
        s512 = timed_steps(model, 512)
        tb512 = token_bytes(512)
        ctx = {"tokens_per_s": round(K * world / s512, 2), "bytes_per_token": tb512,
               "GBps": round(tb512 * K / s512 / 1e9, 1)}

    # ---- M-token sweep of one Q4_K matrix (tensor cores vs one GEMV per token)
    msweep = run_msweep(device) if not args.no_msweep else {}
    lowbit = run_lowbit(device) if not args.no_msweep else {}
    standalone = run_standalone(device) if not args.no_msweep else {}

    out = {
        "metric": METRIC,
        "value": round(tok_s, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(max_s / K * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(tok_s / PAGES_BASELINE_TOK_S, 3),
        "dtype": DTYPE,
        "data": "synthetic (seeded random-init Q4_K/Q6_K weights, N(0,1) hidden inputs)",
        "config": bench_config(world),
        "mode": mode,
        "hbm": {"achieved_GBps_token": round(tb * tok_s / world / 1e9, 1), "peak_GBps": peak,
                "frac_of_peak": round(tb * tok_s / world / 1e9 / peak, 4), "peak_source": peak_src,
                "roofline_tokens_per_s": round(peak * 1e9 / tb, 1)},
        "roofline": {"bound": "hbm", "kernel": rl_kernel, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_src},
        "separate_kernels": separate,
        "ctx512": ctx,
        "msweep": msweep,
        "lowbit_gemv": lowbit,
        "standalone": standalone,
        "e2e": {"value": round(K * world / e2e_max, 2), "unit": "tokens/s", "h2d_bytes_per_step": 4 * m.hidden,
                "d2h_bytes_per_step": 4 * m.vocab},
        "gpu_launches": model.launches_per_step * K,
        "clocks": clocks.summary(),
        "device_error_flag": err,
        "setup_s": round(setup_s, 1),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(m)
    if rank == 0:
        print(json.dumps(out), flush=True)
    model.close()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


SWEEP_ROWS, SWEEP_K = 12288, 4096
SWEEP_M = (1, 2, 4, 8, 16, 64)


def run_msweep(device, reps: int = 20) -> dict:
    """Y[M x 12288] = X[M x 4096] W^T over one Q4_K matrix for M in SWEEP_M, both
    paths, each call on the next of enough device copies of W to exceed L2
    (every call reads W from HBM).  Time per call from CUDA events."""
    import torch

    from quantised_gemv_norm_gb300 import dq

    W = torch.from_numpy(synth.quant_matrix(SEED, synth.FMT_Q4K, SWEEP_ROWS, SWEEP_K)).to(device)
    wbytes = W.numel()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    copies = [W] + [W.clone() for _ in range(max(1, (3 * l2) // wbytes))]
    X = torch.from_numpy(np.stack([synth.activation(SEED, SWEEP_K, m) for m in range(max(SWEEP_M))])).to(device)
    Y = torch.empty((max(SWEEP_M), SWEEP_ROWS), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    out = {"rows": SWEEP_ROWS, "K": SWEEP_K, "weight_bytes": wbytes, "copies_rotated": len(copies)}
    ws = dq.matmul_split_workspace(max(SWEEP_M), SWEEP_ROWS, SWEEP_K, device)

    def call(path, Wc, Xm, Ym):
        if path is None:  # tensor cores, K split across blocks
            dq.matmul_q4k_split(Wc, Xm, ws, out=Ym)
        else:
            dq.matmul_q4k(Wc, Xm, out=Ym, path=path)

    for name, path in (("tensor_split", None), ("tensor", dq.MATMUL_TENSOR), ("cuda_core", dq.MATMUL_CUDA_CORE)):
        res = {}
        for M in SWEEP_M:
            Xm, Ym = X[:M], Y[:M]
            for i in range(3):
                call(path, copies[i % len(copies)], Xm, Ym)
            torch.cuda.synchronize(device)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(20_000_000)  # the calls queue behind it: the events time the GPU
            a.record(stream)
            for i in range(reps):
                call(path, copies[i % len(copies)], Xm, Ym)
            b.record(stream)
            torch.cuda.synchronize(device)
            us = a.elapsed_time(b) * 1e3 / reps
            res[str(M)] = {"us": round(us, 2), "GBps": round(wbytes / us / 1e3, 1),
                           "TFLOPs": round(2.0 * M * SWEEP_ROWS * SWEEP_K / us / 1e6, 2)}
        out[name] = res
    R, rsrc = tensor_peak_tflops()
    bw, bsrc = hbm_peak_gbs()
    out["predicted_M_star"] = round(ledger.m_star(4.5, R * 1e12, bw * 1e9), 1)
    out["M_star_inputs"] = {"R_TFLOPs": R, "R_source": rsrc, "BW_GBps": bw, "BW_source": bsrc}
    t1 = out["tensor"]["1"]["us"]
    out["tensor_cost_ratio_vs_M1"] = {k: round(v["us"] / t1, 3) for k, v in out["tensor"].items()}
    t1 = out["tensor_split"]["1"]["us"]
    out["tensor_split_cost_ratio_vs_M1"] = {k: round(v["us"] / t1, 3) for k, v in out["tensor_split"].items()}
    return out


def graph_us(fn, n: int, device) -> float:
    """Per-call time of n calls fn(0..n-1) captured in one CUDA graph and replayed
    (the launch cost of a captured chain instead of a stream's); CUDA events around
    one replay, after three warm replays."""
    import torch

    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        fn(0)  # any first-call set-up happens outside the capture
        torch.cuda.synchronize(device)
        with torch.cuda.graph(g, stream=side):
            for i in range(n):
                fn(i)
    torch.cuda.synchronize(device)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize(device)
    del g
    return a.elapsed_time(b) * 1e3 / n


def run_lowbit(device, reps: int = 20) -> dict:
    """The 2-bit (Q2_K) GEMV against the 4- and 6-bit ones on the same shapes:
    per call time from CUDA events, each call on the next of enough device
    copies to exceed L2 (weights read from HBM every call)."""
    import torch

    from quantised_gemv_norm_gb300 import dq

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    stream = torch.cuda.current_stream(device)
    bw, bsrc = hbm_peak_gbs()
    out = {}
    for rows, K in ((12288, 4096), (151936, 4096)):
        x = torch.from_numpy(synth.activation(SEED, K)).to(device)
        y = torch.empty(rows, dtype=torch.float32, device=device)
        res = {}
        for name, fmt, fn in (("q2k", synth.FMT_Q2K, dq.gemv_q2k), ("q4k", synth.FMT_Q4K, dq.gemv_q4k),
                              ("q6k", synth.FMT_Q6K, dq.gemv_q6k)):
            W = torch.from_numpy(synth.quant_matrix(SEED, fmt, rows, K)).to(device)
            wbytes = W.numel()
            copies = [W] + [W.clone() for _ in range(max(0, -(-(3 * l2) // wbytes) - 1))]
            for i in range(3):
                fn(copies[i % len(copies)], x, out=y)
            torch.cuda.synchronize(device)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(20_000_000)  # the calls queue behind it: the events time the GPU
            a.record(stream)
            for i in range(reps):
                fn(copies[i % len(copies)], x, out=y)
            b.record(stream)
            torch.cuda.synchronize(device)
            us = a.elapsed_time(b) * 1e3 / reps
            res[name] = {"weight_bytes": wbytes, "us": round(us, 2), "GBps": round(wbytes / us / 1e3, 1),
                         "frac_of_peak": round(wbytes / us / 1e3 / bw, 4), "weights_per_ns": round(rows * K / us / 1e3, 1)}
            if rows < 100000:
                gus = graph_us(lambda i: fn(copies[i % len(copies)], x, out=y), 100, device)
                res[name]["graph_us"] = round(gus, 2)
                res[name]["graph_frac_of_peak"] = round(wbytes / gus / 1e3 / bw, 4)
            del copies, W
        out["%dx%d" % (rows, K)] = res
    out["peak_GBps"] = bw
    out["peak_source"] = bsrc
    return out


def run_standalone(device, reps: int = 20) -> dict:
    """The bf16 GEMV on the shapes of the bf16 configuration (weights larger than L2
    read from HBM each call: enough rotated copies) and the two norms on the
    64x2048 norm configuration, with the default block and with one thread per row
    (the pages' serial norm).  Device-generated seeded inputs; CUDA events."""
    import torch

    from quantised_gemv_norm_gb300 import dq

    stream = torch.cuda.current_stream(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    bw, bsrc = hbm_peak_gbs()
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED)

    def timed(fn, n):
        # the calls queue behind a device-side sleep, so the events time the GPU running
        # them back to back rather than the host issuing them
        for i in range(3):
            fn(i)
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(20_000_000)
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) * 1e3 / n

    out = {"bf16_gemv": {}, "norms": {}}
    for rows, K in ((4096, 4096), (12288, 4096), (4096, 12288), (151936, 4096)):
        W = (torch.randn((rows, K), generator=gen, device=device) * 0.02).to(torch.bfloat16)
        x = torch.randn((K,), generator=gen, device=device).to(torch.bfloat16)
        y = torch.empty(rows, dtype=torch.float32, device=device)
        wbytes = W.numel() * 2
        copies = [W] + [W.clone() for _ in range(max(0, -(-(3 * l2) // wbytes) - 1))]
        us = timed(lambda i: dq.gemv_bf16(copies[i % len(copies)], x, out=y), reps if rows < 100000 else 5)
        out["bf16_gemv"]["%dx%d" % (rows, K)] = {"weight_bytes": wbytes, "us": round(us, 2),
                                                 "GBps": round(wbytes / us / 1e3, 1),
                                                 "frac_of_peak": round(wbytes / us / 1e3 / bw, 4)}
        if rows < 100000:
            gus = graph_us(lambda i: dq.gemv_bf16(copies[i % len(copies)], x, out=y), 100, device)
            out["bf16_gemv"]["%dx%d" % (rows, K)]["graph_us"] = round(gus, 2)
            out["bf16_gemv"]["%dx%d" % (rows, K)]["graph_frac_of_peak"] = round(wbytes / gus / 1e3 / bw, 4)
        del copies, W
    out["bf16_gemv"]["peak_GBps"], out["bf16_gemv"]["peak_source"] = bw, bsrc
    rows, n = 64, 2048
    x = torch.randn((rows, n), generator=gen, device=device)
    g = 1.0 + 0.1 * torch.randn((n,), generator=gen, device=device)
    bt = 0.1 * torch.randn((n,), generator=gen, device=device)
    y = torch.empty_like(x)
    for threads in (None, 1):
        key = "default_block" if threads is None else "one_thread_per_row"
        out["norms"][key] = {
            "rmsnorm_us": round(timed(lambda i: dq.rmsnorm(x, g, 1e-6, out=y, threads=threads), 100), 2),
            "layernorm_us": round(timed(lambda i: dq.layernorm(x, g, bt, 1e-6, out=y, threads=threads), 100), 2),
        }
    out["norms"]["shape"] = "%dx%d fp32" % (rows, n)
    return out


OP_PROBES = ("attention_512", "gemv_bf16_4096", "rmsnorm_default", "rmsnorm_one_thread", "matmul_tensor_m16",
             "matmul_split_m16")


def run_op_probe(args):
    """`probe_reps` launches of one standalone entry point on a small case (for
    profilers): attention over 513 keys of a 32/8-head cache, the bf16 GEMV on
    4096x4096, RMSNorm of 64x2048 with the default block or one thread per row, or
    the tensor-core product of 16 tokens over the 12288x4096 Q4_K table (rows per
    block, or K split across blocks)."""
    import torch

    from quantised_gemv_norm_gb300 import build, dq

    build.build()
    dq.load()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(SEED)
    kind = args.op_probe
    if kind == "attention_512":
        n_q, n_kv, max_ctx, n_keys = 32, 8, 1024, 513
        q = torch.randn((n_q, 128), generator=gen, device="cuda")
        k = torch.randn((n_kv, max_ctx, 128), generator=gen, device="cuda").half()
        v = torch.randn((n_kv, max_ctx, 128), generator=gen, device="cuda").half()
        ws = dq.attention_workspace(n_q, n_kv)
        for _ in range(args.probe_reps):
            y = dq.attention_decode(q, k, v, n_keys, workspace=ws)
    elif kind == "gemv_bf16_4096":
        W = (0.02 * torch.randn((4096, 4096), generator=gen, device="cuda")).to(torch.bfloat16)
        x = torch.randn((4096,), generator=gen, device="cuda").to(torch.bfloat16)
        for _ in range(args.probe_reps):
            y = dq.gemv_bf16(W, x)
    elif kind == "matmul_tensor_m16":
        W = torch.from_numpy(synth.quant_matrix(SEED, synth.FMT_Q4K, SWEEP_ROWS, SWEEP_K)).cuda()
        X = torch.from_numpy(np.stack([synth.activation(SEED, SWEEP_K, m) for m in range(16)])).cuda()
        for _ in range(args.probe_reps):
            y = dq.matmul_q4k(W, X, path=dq.MATMUL_TENSOR)
    elif kind == "matmul_split_m16":
        W = torch.from_numpy(synth.quant_matrix(SEED, synth.FMT_Q4K, SWEEP_ROWS, SWEEP_K)).cuda()
        X = torch.from_numpy(np.stack([synth.activation(SEED, SWEEP_K, m) for m in range(16)])).cuda()
        ws = dq.matmul_split_workspace(16, SWEEP_ROWS, SWEEP_K)
        for _ in range(args.probe_reps):
            y = dq.matmul_q4k_split(W, X, ws)
    else:
        x = torch.randn((64, 2048), generator=gen, device="cuda")
        g = 1.0 + 0.1 * torch.randn((2048,), generator=gen, device="cuda")
        for _ in range(args.probe_reps):
            y = dq.rmsnorm(x, g, 1e-6, threads=None if kind == "rmsnorm_default" else 1)
    torch.cuda.synchronize()
    err = dq.device_error()
    print(json.dumps({"op_probe": kind, "reps": args.probe_reps, "device_error_flag": err,
                      "finite": bool(torch.isfinite(y).all().item())}))
    if err:
        sys.exit(1)


def run_kernel_probe(args):
    """One decode token of a 2-layer full-width stack (9 GEMV launches), then the
    chosen kernel kind on layer 1 (a Q6_K down layer), alone, `probe_reps` times."""
    import torch

    from quantised_gemv_norm_gb300 import build, dq, upload

    build.build()
    dq.load()
    S = synth.QWEN3_8B
    m = synth.make_model(SEED, n_layers=2, hidden=S["hidden"], ffn=S["ffn"], n_q_heads=S["n_q_heads"],
                         n_kv_heads=S["n_kv_heads"], head_dim=S["head_dim"], vocab=S["vocab"], max_ctx=MAX_CTX,
                         qwen3_attention=True)
    w = upload.to_device(m, synth.make_kv_cache(SEED, m, 0))
    model = dq.Model(**upload.model_kwargs(m), weights=w, use_graph=False)
    x = torch.from_numpy(synth.decode_input(SEED, m.hidden)).cuda()
    logits = model.step(x, 0)
    kind = KERNEL_KINDS.index(args.kernel_probe)
    for _ in range(args.probe_reps):
        model.enqueue_kernel(1, kind)
    torch.cuda.synchronize()
    err = dq.device_error()
    model.close()
    print(json.dumps({"kernel_probe": args.kernel_probe, "reps": args.probe_reps, "device_error_flag": err,
                      "logits_finite": bool(torch.isfinite(logits).all().item())}))
    if err:
        sys.exit(1)


def run_token_probe(args):
    """`probe_reps` decode tokens of a 2-layer full-width stack (the Qwen3-8B layer
    shapes and vocabulary, 740 MB of weights) through the fused token kernel: a
    small case of the headline kernel for profilers."""
    import torch

    from quantised_gemv_norm_gb300 import build, dq, upload

    build.build()
    dq.load()
    S = synth.QWEN3_8B
    m = synth.make_model(SEED, n_layers=2, hidden=S["hidden"], ffn=S["ffn"], n_q_heads=S["n_q_heads"],
                         n_kv_heads=S["n_kv_heads"], head_dim=S["head_dim"], vocab=S["vocab"], max_ctx=MAX_CTX,
                         qwen3_attention=True)
    w = upload.to_device(m, synth.make_kv_cache(SEED, m, 0))
    model = dq.Model(**upload.model_kwargs(m), weights=w, flags=dq.MODEL_FUSED)
    x = torch.from_numpy(synth.decode_input(SEED, m.hidden)).cuda()
    for _ in range(args.probe_reps):
        logits = model.step(x, 0)
    torch.cuda.synchronize()
    err = dq.device_error()
    fused = model.fused
    model.close()
    print(json.dumps({"token_probe": "2 layers", "fused": fused, "reps": args.probe_reps,
                      "weight_bytes": int(m.weight_bytes()), "device_error_flag": err,
                      "logits_finite": bool(torch.isfinite(logits).all().item())}))
    if err or not fused:
        sys.exit(1)


# -------------------------------------------------------------- the oracle


def cpu_baseline(m, budget_s: float = 10.0, max_tokens: int = 30):
    """The fp64 CPU oracle, as it stands, on this host's cores: full decode tokens of
    the same workload until about `budget_s` seconds of CPU work (at least one)."""
    import oracle

    oracle.build()
    kv = synth.make_kv_cache(SEED, m, 0)
    t0 = time.perf_counter()
    tokens = 0
    while tokens < max_tokens and (tokens == 0 or time.perf_counter() - t0 < budget_s):
        oracle.decode_step(m, synth.decode_input(SEED, m.hidden, tokens), 0, kv)
        tokens += 1
    dt = time.perf_counter() - t0
    return {"value": round(tokens / dt, 4), "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d full decode token(s) of the same workload (pos 0), fp64, %.1f s" % (tokens, dt)}


REFERENCE_BUDGET_S = 120.0  # host seconds the reference arm's timed steps may take


def sample_model(m, n_layers: int, vocab: int):
    """The first `n_layers` layers and `vocab` vocabulary rows of `m`: a bounded
    sample of the same workload (every layer keeps its shapes and formats)."""
    import dataclasses

    per_layer = ("attn_norm", "wqkv", "wo", "ffn_norm", "wgate", "wup", "wdown", "down_fmt", "q_norm", "k_norm")
    cut = {name: getattr(m, name)[:n_layers] for name in per_layer}
    return dataclasses.replace(m, n_layers=n_layers, vocab=vocab, wvocab=m.wvocab[:vocab], **cut)


def run_reference(args):
    """The oracle as the reference arm: --steps K timed steps after --warmup W, each
    step one decode token on the host cores.  When K full tokens would take longer
    than REFERENCE_BUDGET_S (measured on the first warm-up token), each step is the
    same fraction of the token instead -- its first layers and vocabulary rows, in
    proportion -- and tokens/s counts that fraction of a token per step (by weight
    bytes, which set the oracle's work)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    m = synth.make_model(SEED, max_ctx=MAX_CTX, qwen3_attention=True, **synth.QWEN3_8B)
    import oracle

    oracle.build()
    full_bytes = m.weight_bytes()
    t0 = time.perf_counter()
    oracle.decode_step(m, synth.decode_input(SEED, m.hidden, 0), 0, synth.make_kv_cache(SEED, m, 0))
    t_token = time.perf_counter() - t0
    frac = min(1.0, REFERENCE_BUDGET_S / (args.steps * t_token))
    s = m if frac >= 1.0 else sample_model(m, max(1, int(m.n_layers * frac)), max(1, int(m.vocab * frac)))
    share = s.weight_bytes() / full_bytes
    kv = synth.make_kv_cache(SEED, s, 0)
    for t in range(1, args.warmup):
        oracle.decode_step(s, synth.decode_input(SEED, s.hidden, t), 0, kv)
    t0 = time.perf_counter()
    for t in range(args.steps):
        oracle.decode_step(s, synth.decode_input(SEED, s.hidden, args.warmup + t), 0, kv)
    dt = time.perf_counter() - t0
    v = args.steps * share / dt
    cores = oracle.num_threads()
    if s is m:
        sample = "%d full decode tokens on the host, fp64" % args.steps
    else:
        sample = ("%d steps, each the first %d of %d layers and %d of %d vocabulary rows of the token "
                  "(%.4f of its weight bytes), fp64; a full token took %.2f s" %
                  (args.steps, s.n_layers, m.n_layers, s.vocab, m.vocab, share, t_token))
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 4),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(v / PAGES_BASELINE_TOK_S, 5),
        "dtype": "f64",
        "data": "synthetic (seeded random-init Q4_K/Q6_K weights, N(0,1) hidden inputs)",
        "config": bench_config(world),
        "mode": "fp64 CPU oracle on the host cores",
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--no-ctx512", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fused", action="store_true",
                    help="time the separate-kernel CUDA graph as the headline instead of the fused token kernel")
    ap.add_argument("--no-msweep", action="store_true", help="skip the M-token sweep")
    ap.add_argument("--msweep-only", action="store_true", help="print only the M-token sweep")
    ap.add_argument("--kernel-probe", choices=KERNEL_KINDS, default=None,
                    help="profiling aid: build a 2-layer full-width stack, run one token, then launch this "
                         "kernel kind alone --probe-reps times (for ncu -k ... -s 9 -c 1)")
    ap.add_argument("--op-probe", choices=OP_PROBES, default=None,
                    help="profiling aid: launch one standalone entry point on a small case --probe-reps times")
    ap.add_argument("--probe-reps", type=int, default=3)
    ap.add_argument("--token-probe", action="store_true",
                    help="run a few fused tokens of a 2-layer full-width stack (for profilers) and exit")
    args = ap.parse_args()
    if args.token_probe:
        run_token_probe(args)
        return
    if args.kernel_probe:
        run_kernel_probe(args)
        return
    if args.op_probe:
        run_op_probe(args)
        return
    if args.msweep_only:
        import torch

        from quantised_gemv_norm_gb300 import build, dq

        build.build()
        dq.load()
        print(json.dumps({"msweep": run_msweep(torch.device("cuda", 0))}), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
