#!/usr/bin/env python
"""Benchmark of the GB300 Mesa layer forward pass (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl mesa|reference]

A step is one pass of the hot path over one batch of seeded synthetic input: for the forward
workloads one mesa_forward_chunked call (log-decays, chunk states, chunk-level scan, batched
per-token CG with the fused readout); for the decode workload one mesa_decode_step over all
sequences and heads; for the backward workload one mesa_backward_chunked call (the forward's
solves recomputed, the second solve per token, the state adjoints and every gradient).  Inputs are resident in HBM before the timed region; the L2 (129 MB) is
flushed by a 256 MiB device write between timed steps unless the step's working set is
larger than L2.  Kernel times come from CUDA events on the launching stream; `e2e` repeats
the measurement through the same C-ABI call with pinned host buffers, every step's host-to-
device upload of its inputs and download of its results inside the timed region (uploads
double-buffered on a second stream, so that step i+1's upload overlaps step i's compute).
Under torchrun every rank runs its own replica (independent sequences, no collective) and
`value` is the aggregate over ranks with the max-over-ranks time.

`--impl reference` times the fp64 CPU oracle (the deliberately slow restatement of the
method used by the tests) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mesa_layer_gb300 import synth  # noqa: E402

METRIC = "Mesa-layer fwd tokens/s on 1 GB300 (per CG iters) + % tensor/HBM roofline"
METRIC_BWD = "Mesa-layer bwd (all gradients) tokens/s on 1 GB300 (per CG iters) + % roofline of the top kernel"
# the largest configuration that fits one GPU: B=1, 16 heads, T=65536, d=128, bf16, dynamic CG
DEFAULT_WORKLOAD = "long_bf16_d128"
FP32_LANES_PER_SM = 128
ORACLE_MAX_T = 8192  # the CPU oracle's timed sample takes at most this many tokens per unit
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=synth.WORKLOAD_ORDER)
    p.add_argument("--impl", default="mesa", choices=["mesa", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--batch", type=int, default=None,
                   help="override the workload's batch B (small cases for profiler captures; not a bench line)")
    p.add_argument("--decode-prefix", type=int, default=None,
                   help="decode workload: state-only prefix steps (default: the workload's)")
    return p.parse_args()


def source_digest(files) -> str:
    """sha256 over the named library source files (paths relative to the repository)."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode())
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu record, or None
    when there is none or the kernel's sources changed since it was taken (each entry names
    the files its kernel is built from and their sha256)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    entry = rec.get("workloads", {}).get(workload)
    if not entry or entry.get("kernel") != kernel:
        return None
    try:
        if source_digest(entry["sources"]) != entry.get("sources_sha256"):
            return None
    except (KeyError, OSError):
        return None
    return entry.get("dram_bytes_per_launch")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


# ------------------------------------------------------------------------------------------
# algorithmic work (what the method must compute; causal half of the chunk blocks)


def cg_flops(w, iters: np.ndarray) -> float:
    """Per token-head and CG iteration: the matrix-vector product with H_t + Lambda in
    chunk form, 2 d^2 (state term) + 2 d (C + 1) (causal intra-chunk term, both products);
    the readout costs one more such product.  iters holds each token's own count."""
    d, C = w.dk, w.chunk
    per = 2.0 * d * d + 2.0 * d * (C + 1)
    return float((iters.astype(np.float64) + 1.0).sum() * per)


def tc_executed_flops(w, iters: np.ndarray, readout: bool = True) -> float:
    """MMA flops the tensor-core CG kernels issue per 128-token chunk and iteration: d = 128
    (bf16 inputs) 7 products of 128x128x128 (3 for the split state product, 2 + 2 for the key
    products); d = 64 (fp32 inputs, keys split too) 3 x (128x128x64 + 128x64x64 + 128x64x128);
    iterations run until the slowest token of the chunk stops, plus the readout."""
    B, H, T = iters.shape
    nc = (T + 127) // 128
    pad = np.zeros((B, H, nc * 128), dtype=np.int64)
    pad[:, :, :T] = iters
    per_chunk = pad.reshape(B, H, nc, 128).max(axis=-1) + (1 if readout else 0)
    if w.dk == 64:
        per = 3 * 2.0 * (128 * 128 * 64 + 128 * 64 * 64 + 128 * 64 * 128)
    else:
        per = 7 * 2.0 * 128 ** 3
    return float(per_chunk.sum()) * per


def state_flops(w) -> float:
    """Chunk-local state sums: 2 d^2 multiply-adds per token for H and for G."""
    return float(w.B * w.H * w.T) * 4.0 * w.dk * w.dk


def bwd_grad_flops(w, states_apart: bool = False) -> float:
    """The gradient kernel per token-head (32-token chunks, causal halves): the three C x C
    dot-product blocks G V^T, X K^T, Y K^T (3 d (C + 1)), the four intra-chunk products with
    them (4 d (C + 1)) and six d x d products with the chunk states and state adjoints
    (12 d^2) -- unless those products come from the tensor-core kernel (states_apart)."""
    d, C = w.dk, 32
    return float(w.B * w.H * w.T) * ((0.0 if states_apart else 12.0 * d * d) + 7.0 * d * (C + 1))


def bwd_sprod_flops(w) -> float:
    """The tensor-core products of the backward's rows with the chunk states, per token-head:
    dG k, dG^T v, dH k, dH^T k, S^H x (2 d^2 each)."""
    return float(w.B * w.H * w.T) * 10.0 * w.dk * w.dk


def bwd_sprod_executed_flops(w) -> float:
    """MMA flops that kernel issues per 32-token chunk: 88 products of 128 x 32 x 16 (the
    states split hi + lo, x split as well: 16 + 16 + 32 + 24)."""
    nc = w.B * w.H * ((w.T + 31) // 32)
    return float(nc) * 88 * 2.0 * 128 * 32 * 16


def bwd_rhs_flops(w) -> float:
    """b = G_t^T g_t in chunk form: 2 d^2 + 2 d (C + 1) per token-head."""
    d, C = w.dk, 32
    return float(w.B * w.H * w.T) * (2.0 * d * d + 2.0 * d * (C + 1))


def preprocess_bytes(w) -> float:
    """Raw q and k read once, preprocessed q and k written once, plus the taps."""
    esz = 2 if w.dtype == "bf16" else 4
    return float(w.B * w.H * w.T * w.dk) * esz * 2 * 2 + 2.0 * w.H * w.dk * w.conv_taps * 4


def decode_bytes(w) -> float:
    """Per unit and step: H and G read and written in fp32, plus q, k, v, gamma, out, iters."""
    esz = 2 if w.dtype == "bf16" else 4
    U = w.B * w.H
    warm = 2 * 4 * w.dk if w.warm else 0  # the start vector read and written
    return float(U) * (2 * 4 * (w.dk * w.dk + w.dv * w.dk) + esz * (2 * w.dk + 2 * w.dv) + 4 + 4 + warm)


# ------------------------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.device_id = device_id
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.device_id:
            cmd += ["-i", self.device_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def device_id_for_smi(torch, dev):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


# ------------------------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)


def oracle_sample(w, budget_s: float = 20.0):
    """Time the fp64 oracle on a bounded sample of the workload: a subset of (batch, head)
    units (forward) or of (sequence, head) units over a few steps (decode).  Returns
    (tokens per second, threads used, description, seconds)."""
    import oracle

    threads = oracle.max_threads()
    if w.conv_taps and not w.fused:
        units = min(w.B * w.H, 8)
        inp = synth.preprocess_inputs(synth.workload(w.name, B=1, H=units))
        total, dt, passes = 0, 0.0, 0
        while dt < budget_s / 4 or passes == 0:
            t0 = time.perf_counter()
            oracle.qk_preprocess(inp["q_raw"], inp["wq"])
            oracle.qk_preprocess(inp["k_raw"], inp["wk"])
            dt += time.perf_counter() - t0
            total += units * w.T
            passes += 1
        return total / dt / w.H, 1, f"{passes} pass(es) over {units} (batch, head) units x {w.T} tokens, q and k", dt
    if w.backward:
        # whole units: the fp64 backward per unit (two solves per token and the adjoint sweep)
        n_units = min(w.B * w.H, max(1, threads))
        sub = synth.backward_inputs(synth.workload(w.name, B=1, H=n_units))
        total, dt, passes = 0, 0.0, 0
        while dt < budget_s / 2 or passes == 0:
            t0 = time.perf_counter()
            oracle.backward(sub["q"], sub["k"], sub["v"], sub["gamma"], sub["lam"], sub["dout"], w.cg_iters,
                            w.cg_tol, nthreads=threads)
            dt += time.perf_counter() - t0
            total += n_units * w.T
            passes += 1
        return total / dt / w.H, min(threads, n_units), f"{passes} pass(es) over {n_units} (batch, head) units x {w.T} tokens", dt
    if w.decode_steps:
        units = min(w.B * w.H, 64 * max(1, threads))
        steps = 8
        inp = synth.decode_inputs(w, 0)
        q = inp["q"].reshape(1, -1, w.dk)[:, :units]
        k = inp["k"].reshape(1, -1, w.dk)[:, :units]
        v = inp["v"].reshape(1, -1, w.dv)[:, :units]
        g = inp["gamma"].reshape(1, -1)[:, :units]
        lam = synth.lambdas(w)[np.arange(units) % w.H]  # unit i keeps its head's lambda
        Hs = np.zeros((1, units, w.dk, w.dk))
        Gs = np.zeros((1, units, w.dv, w.dk))
        X = np.zeros((1, units, w.dk)) if w.warm else None
        t0 = time.perf_counter()
        for _ in range(steps):
            oracle.decode_step(Hs, Gs, q, k, v, g, lam, w.cg_iters, w.cg_tol, nthreads=threads, X=X)
        dt = time.perf_counter() - t0
        return units * steps / dt / w.H, min(threads, units), f"{units} (sequence, head) units x {steps} steps", dt
    # forward: whole units (sequences are sequential in t); the unit count grows until one
    # pass takes a good part of the budget, then passes repeat until the budget is used
    # a long sequence is sampled as its first ORACLE_MAX_T tokens (the oracle's cost per
    # token does not depend on the position)
    T = min(w.T, ORACLE_MAX_T)
    full = synth.forward_inputs(w) if w.B * w.H * w.T <= (1 << 22) and T == w.T else None
    U = w.B * w.H
    n_units = min(U, max(1, threads))
    total_th, total_t, passes = 0, 0.0, 0
    while True:
        if full is not None:
            sub = {k: full[k].reshape((U,) + full[k].shape[2:])[:n_units][None] for k in ("q", "k", "v", "gamma")}
            lam = full["lam"][np.arange(n_units) % w.H]
        else:
            sub = synth.forward_inputs(synth.workload(w.name, B=1, H=n_units, T=T))
            lam = sub["lam"]
        pre = synth.preprocess_inputs(synth.workload(w.name, B=1, H=n_units, T=T)) if w.fused else None
        t0 = time.perf_counter()
        if pre is not None:  # the preprocessing, then the layer (rounded to the dtype between)
            sub["q"] = synth.round_bf16(oracle.qk_preprocess(pre["q_raw"], pre["wq"]).astype(np.float32))
            sub["k"] = synth.round_bf16(oracle.qk_preprocess(pre["k_raw"], pre["wk"]).astype(np.float32))
        oracle.forward(sub["q"], sub["k"], sub["v"], sub["gamma"], lam, w.cg_iters, w.cg_tol, nthreads=threads)
        dt = time.perf_counter() - t0
        if n_units < U and dt < 0.25 * budget_s:
            n_units = min(U, n_units * 2)
            continue
        total_th += n_units * T
        total_t += dt
        passes += 1
        if total_t >= budget_s or dt > budget_s / 2:
            break
    desc = f"{passes} pass(es) over {n_units} (batch, head) units x {T} tokens" + (
        f" (the first {T} of each unit's {w.T})" if T < w.T else "")
    # tokens/s of the workload = token-heads/s divided by the heads per token
    return total_th / total_t / w.H, min(threads, n_units), desc, total_t


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = synth.workload(args.workload)
    import oracle
    oracle.load()
    vals = []
    desc = ""
    cores = 1
    for _ in range(max(1, args.steps)):
        v, cores, desc, _ = oracle_sample(w, budget_s=min(15.0, 120.0 / max(1, args.steps)))
        vals.append(v)
    value = statistics.median(vals)
    unit = "tokens/s"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def arithmetic(w) -> str:
    """What the timed path computes in, for the line's config."""
    if w.conv_taps and not w.fused:
        return f"{w.dtype} in and out, fp32 convolution and norm"
    if w.decode_steps:
        return f"{w.dtype} q/k/v, fp32 states and CG (CUDA cores)"
    if w.dtype == "bf16" and w.dk == 128:
        return (("raw q, k preprocessed in fp32 and rounded to bf16 in the prologues; " if w.fused else "") +
                "bf16 inputs; tensor-core products of fp16 hi+lo split operands with fp32 "
                "accumulation; fp32 CG vectors and scalars")
    if w.dtype == "f32" and w.dk == 64:
        return ("fp32 inputs; tensor-core products of fp16 hi+lo split operands (keys and values split "
                "too) with fp32 accumulation; fp32 chunk states (CUDA cores), CG vectors and scalars")
    return f"{w.dtype} inputs, fp32 CUDA-core arithmetic"


def workload_config(w, extra=None):
    cfg = {"workload": w.name, "B": w.B, "heads": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
           "chunk": w.chunk, "qkv_dtype": w.dtype,
           "cg": (f"dynamic tol {w.cg_tol:g}, max {w.cg_iters}" if w.cg_tol > 0 else f"fixed {w.cg_iters}"),
           "parallelism": "replicas"}
    if w.decode_steps:
        cfg.update({"sequences": w.B, "decode_steps": w.decode_steps, "prefix": w.prefix})
        cfg.pop("T")
        if w.warm:
            cfg["cg"] += ", warm start from the previous step's solution"
    if w.backward:
        cfg["step"] = ("backward given the forward's kept iterates: second CG per token on G_t^T dout_t, "
                       "chunk states and state adjoints, dq/dk/dv/dgamma/dlambda")
        cfg["chunk"] = "32 (gradient kernels), 128 (tensor-core solves)"
    if w.fused:
        cfg["conv_taps"] = w.conv_taps
        cfg["step"] = (f"query/key preprocessing (causal depthwise conv, {w.conv_taps} taps, + L2 norm) fused "
                       "into the forward's prologues, then the layer")
    elif w.conv_taps:
        cfg = {"workload": w.name, "B": w.B, "heads": w.H, "T": w.T, "d": w.dk, "qk_dtype": w.dtype,
               "conv_taps": w.conv_taps, "step": "q/k preprocessing: causal depthwise conv + L2 norm",
               "parallelism": "replicas"}
    cfg.update(extra or {})
    return cfg


# ------------------------------------------------------------------------------------------
# GPU arm


def kind_names(lib):
    names = []
    for i in range(16):
        n = lib.mesa_kernel_name(i)
        if n is None:
            break
        names.append(n.decode())
    return names


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    w = synth.workload(args.workload, **({"B": args.batch} if args.batch else {}))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_sample(w, budget_s=10.0)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}

    import torch
    import torch.distributed as dist

    from mesa_layer_gb300 import binding, build

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    build.build()
    lib = binding.load()
    lib.mesa_kernel_name.restype = ctypes.c_char_p
    lib.mesa_kernel_name.argtypes = [ctypes.c_int]
    lib.mesa_timing_begin.argtypes = [ctypes.c_int]
    lib.mesa_timing_end.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    names = kind_names(lib)
    dev = torch.device("cuda", local)
    peaks = measured_peaks()
    peaks["sm_count"] = torch.cuda.get_device_properties(dev).multi_processor_count
    if w.conv_taps and not w.fused:
        res = bench_preprocess(args, w, rank, world, dev, lib, torch, binding)
    elif w.backward:
        res = bench_backward(args, w, rank, world, dev, lib, torch, binding)
    elif w.decode_steps:
        res = bench_decode(args, w, rank, world, dev, lib, torch, binding)
    else:
        res = bench_forward(args, w, rank, world, dev, lib, torch, binding)
    res["names"] = names
    emit(args, w, res, peaks, cpu, rank, world, torch, dist)
    if world > 1:
        dist.destroy_process_group()


def timed_loop(args, torch, lib, step_fn, flush_fn, world, dist, dev):
    """W warm-up steps, then K steps each bracketed by CUDA events (flush outside)."""
    for i in range(args.warmup):
        step_fn(i)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    nk = 16
    ms_kind = (ctypes.c_double * nk)()
    n_kind = (ctypes.c_int * nk)()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(device_id_for_smi(torch, dev.index)).start()
    time.sleep(0.3)
    assert lib.mesa_timing_begin(8 * args.steps + 8) == 0
    t_wall = time.perf_counter()
    for i in range(args.steps):
        if flush_fn is not None:
            flush_fn()
        starts[i].record()
        step_fn(i)
        ends[i].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    assert lib.mesa_timing_end(ms_kind, n_kind, nk) == 0
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return {"step_ms": step_ms, "kind_ms": list(ms_kind), "kind_n": list(n_kind), "wall_s": wall,
            "clocks": clocks}


def bench_forward(args, w, rank, world, dev, lib, torch, binding):
    import torch.distributed as dist
    inp = synth.forward_inputs(w, seed=rank)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    if w.fused:  # raw queries and keys with their taps in place of q and k
        pre = synth.preprocess_inputs(w, seed=rank)
        inp["q"], inp["k"] = pre["q_raw"], pre["k_raw"]
        inp["wq"], inp["wk"] = pre["wq"], pre["wk"]
    d_in = {k: torch.from_numpy(inp[k]).to(dev).to(td if k in ("q", "k", "v") else torch.float32).contiguous()
            for k in ("q", "k", "v", "gamma", "lam") + (("wq", "wk") if w.fused else ())}
    out = torch.empty((w.B, w.H, w.T, w.dv), dtype=td, device=dev)
    iters = torch.empty((w.B, w.H, w.T), dtype=torch.int32, device=dev)
    ws = torch.empty(binding.mesa_forward_pre_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.chunk,
                                                             1 if w.dtype == "bf16" else 0),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    in_bytes = sum(d_in[k].numel() * d_in[k].element_size() for k in ("q", "k", "v", "gamma"))
    needs_flush = in_bytes < 2 * (129 << 20)

    def step(i):
        if w.fused:
            binding.mesa_forward_chunked_pre(d_in["q"], d_in["k"], d_in["wq"], d_in["wk"], d_in["v"], d_in["gamma"],
                                             d_in["lam"], w.cg_iters, w.cg_tol, w.chunk, out=out, iters_used=iters,
                                             workspace=ws)
        else:
            binding.mesa_forward_chunked(d_in["q"], d_in["k"], d_in["v"], d_in["gamma"], d_in["lam"],
                                         w.cg_iters, w.cg_tol, w.chunk, out=out, iters_used=iters, workspace=ws)

    res = timed_loop(args, torch, lib, step, (lambda: flush.random_(0, 255)) if needs_flush else None,
                     world, dist, dev)
    it = iters.cpu().numpy()
    res.update({"iters": it, "tokens_per_step": w.B * w.T, "flush": needs_flush})
    if not args.no_e2e:
        res["e2e"] = e2e_forward(args, w, dev, torch, binding, inp, td, ws)
    return res


def pipelined_e2e(torch, dev, host_in, run, host_out: dict, steps: int, warmup: int = 3):
    """Time `steps` end-to-end steps: each copies its inputs from pinned host memory to the
    device, runs the call, and copies its results back to pinned host memory.  Inputs and
    results are double-buffered on the device, uploads and downloads run on streams of their
    own, so that step i+1's upload and step i-1's download overlap step i's compute (as a
    caller streaming batches would run it).  `host_in` is a dict of pinned tensors, or a list
    of them used in turn.  `run(d_in, stream, slot)` launches the call on `stream` with its
    results in device buffer set `slot` (0 or 1) and returns them, matched by name to
    `host_out`.  Returns ms per step (first upload issued to last download done)."""
    ins = host_in if isinstance(host_in, list) else [host_in]
    s_up, s_comp, s_down = (torch.cuda.Stream(device=dev) for _ in range(3))
    bufs = [{k: torch.empty_like(v, device=dev) for k, v in ins[0].items()} for _ in range(2)]
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    in_ready, in_free, out_ready, out_free = ev(), ev(), ev(), ev()
    for e in in_free + out_free:
        e.record(s_comp)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for i in range(warmup + steps):
        b = i % 2
        if i == warmup:
            torch.cuda.synchronize()
            start.record(s_up)
        with torch.cuda.stream(s_up):
            s_up.wait_event(in_free[b])  # the compute that read this input buffer is done
            for k, v in ins[i % len(ins)].items():
                bufs[b][k].copy_(v, non_blocking=True)
            in_ready[b].record(s_up)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_ready[b])
            s_comp.wait_event(out_free[b])  # the download of this result buffer is done
            out = run(bufs[b], s_comp, b)
            in_free[b].record(s_comp)
            out_ready[b].record(s_comp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(out_ready[b])
            for k, v in host_out.items():
                v.copy_(out[k], non_blocking=True)
            out_free[b].record(s_down)
    s_down.wait_stream(s_up)
    s_down.wait_stream(s_comp)
    end.record(s_down)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def e2e_forward(args, w, dev, torch, binding, inp, td, ws):
    """Same call through the C ABI with pinned host buffers: H2D of q, k, v, gamma and D2H of
    out and iters_used inside the timed region of every step (uploads double-buffered)."""
    h = {k: torch.from_numpy(inp[k]).to(td if k in ("q", "k", "v") else torch.float32).pin_memory()
         for k in ("q", "k", "v", "gamma")}
    lam = torch.from_numpy(inp["lam"]).to(dev)
    outs = [{"out": torch.empty((w.B, w.H, w.T, w.dv), dtype=td, device=dev),
             "iters": torch.empty((w.B, w.H, w.T), dtype=torch.int32, device=dev)} for _ in range(2)]
    h_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs[0].items()}
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())

    taps = {k: torch.from_numpy(inp[k]).to(dev) for k in ("wq", "wk")} if w.fused else None

    def run(d, stream, slot):
        o = outs[slot]
        if taps is not None:
            binding.mesa_forward_chunked_pre(d["q"], d["k"], taps["wq"], taps["wk"], d["v"], d["gamma"], lam,
                                             w.cg_iters, w.cg_tol, w.chunk, out=o["out"], iters_used=o["iters"],
                                             workspace=ws, stream=stream)
        else:
            binding.mesa_forward_chunked(d["q"], d["k"], d["v"], d["gamma"], lam, w.cg_iters, w.cg_tol, w.chunk,
                                         out=o["out"], iters_used=o["iters"], workspace=ws, stream=stream)
        return o

    ms = pipelined_e2e(torch, dev, h, run, h_out, max(3, min(args.steps, 50)), max(3, args.warmup))
    return {"ms_per_step": ms, "h2d": h2d, "d2h": d2h}


def bench_decode(args, w, rank, world, dev, lib, torch, binding):
    import torch.distributed as dist
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    N, H, d = w.B, w.H, w.dk
    lam = torch.from_numpy(synth.lambdas(w)).to(dev)
    Hs = torch.zeros(N, H, d, d, device=dev)
    Gs = torch.zeros(N, H, w.dv, d, device=dev)
    Xs = torch.zeros(N, H, d, device=dev) if w.warm else None
    out = torch.empty(N, H, w.dv, dtype=td, device=dev)

    def decode(q, k, v, g):
        if Xs is not None:
            binding.mesa_decode_step_warm(Hs, Gs, Xs, q, k, v, g, lam, w.cg_iters, w.cg_tol, out=out, iters_used=iters)
        else:
            binding.mesa_decode_step(Hs, Gs, q, k, v, g, lam, w.cg_iters, w.cg_tol, out=out, iters_used=iters)
    iters = torch.empty(N, H, dtype=torch.int32, device=dev)

    def dev_inputs(s):
        inp = synth.decode_inputs(w, s, seed=rank)
        return {k: torch.from_numpy(inp[k]).to(dev).to(td if k != "gamma" else torch.float32) for k in inp}

    prefix = w.prefix if args.decode_prefix is None else args.decode_prefix
    for s in range(-prefix, 0):  # state-only prefix (untimed): cg_iters = 0
        x = dev_inputs(s)
        binding.mesa_decode_step(Hs, Gs, x["q"], x["k"], x["v"], x["gamma"], lam, 0, 0.0, out=out, iters_used=iters)
    n_steps = min(w.decode_steps, max(args.steps, 1))
    steps = [dev_inputs(s) for s in range(n_steps)]
    torch.cuda.synchronize()

    def step(i):
        x = steps[i % n_steps]
        decode(x["q"], x["k"], x["v"], x["gamma"])

    res = timed_loop(args, torch, lib, step, None, world, dist, dev)
    res.update({"iters": iters.cpu().numpy(), "tokens_per_step": N, "flush": False})
    if not args.no_e2e:
        hs = [{k: st_[k].cpu().pin_memory() for k in st_} for st_ in steps]
        douts = [{"out": torch.empty_like(out), "iters": torch.empty_like(iters)} for _ in range(2)]
        h_back = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in douts[0].items()}

        def run(d, stream, slot):
            o = douts[slot]
            if Xs is not None:
                binding.mesa_decode_step_warm(Hs, Gs, Xs, d["q"], d["k"], d["v"], d["gamma"], lam, w.cg_iters,
                                              w.cg_tol, out=o["out"], iters_used=o["iters"], stream=stream)
            else:
                binding.mesa_decode_step(Hs, Gs, d["q"], d["k"], d["v"], d["gamma"], lam, w.cg_iters, w.cg_tol,
                                         out=o["out"], iters_used=o["iters"], stream=stream)
            return o

        # each step's own inputs from pinned host memory, in the same order as the device loop
        # (repeating one step's inputs would hand the warm start its own solution)
        ms = pipelined_e2e(torch, dev, hs, run, h_back, max(3, min(args.steps, 50)))
        res["e2e"] = {"ms_per_step": ms, "h2d": sum(t.numel() * t.element_size() for t in hs[0].values()),
                      "d2h": sum(t.numel() * t.element_size() for t in h_back.values())}
    return res


def bench_preprocess(args, w, rank, world, dev, lib, torch, binding):
    import torch.distributed as dist
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inp = synth.preprocess_inputs(w, seed=rank)
    d_in = {k: torch.from_numpy(v).to(dev).to(td if k.endswith("_raw") else torch.float32).contiguous()
            for k, v in inp.items()}
    qo, ko = torch.empty_like(d_in["q_raw"]), torch.empty_like(d_in["k_raw"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    in_bytes = sum(d_in[k].numel() * d_in[k].element_size() for k in ("q_raw", "k_raw"))
    needs_flush = in_bytes < 2 * (129 << 20)

    def step(i):
        binding.mesa_qk_preprocess(d_in["q_raw"], d_in["k_raw"], d_in["wq"], d_in["wk"], q_out=qo, k_out=ko)

    res = timed_loop(args, torch, lib, step, (lambda: flush.random_(0, 255)) if needs_flush else None,
                     world, dist, dev)
    res.update({"iters": np.zeros(1, dtype=np.int32), "tokens_per_step": w.B * w.T, "flush": needs_flush})
    if not args.no_e2e:
        h = {k: torch.from_numpy(inp[k]).to(td).pin_memory() for k in ("q_raw", "k_raw")}
        back = {"q": torch.empty_like(h["q_raw"]).pin_memory(), "k": torch.empty_like(h["k_raw"]).pin_memory()}
        pouts = [{"q": torch.empty_like(qo), "k": torch.empty_like(ko)} for _ in range(2)]

        def run(d, stream, slot):
            o = pouts[slot]
            binding.mesa_qk_preprocess(d["q_raw"], d["k_raw"], d_in["wq"], d_in["wk"], q_out=o["q"], k_out=o["k"],
                                       stream=stream)
            return o

        ms = pipelined_e2e(torch, dev, h, run, back, max(3, min(args.steps, 50)))
        nb = sum(t.numel() * t.element_size() for t in h.values())
        res["e2e"] = {"ms_per_step": ms, "h2d": nb, "d2h": nb}
    return res


def bench_backward(args, w, rank, world, dev, lib, torch, binding):
    """One step = one mesa_backward_chunked call given the forward's kept iterates (as in
    training: mesa_forward_chunked_save runs once, untimed, before the loop); the call that
    recomputes the forward's solves itself is timed as well and reported in config."""
    import torch.distributed as dist
    inp = synth.backward_inputs(w, seed=rank)
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    keys = ("q", "k", "v", "gamma", "dout")
    d_in = {k: torch.from_numpy(inp[k]).to(dev).to(td if k in ("q", "k", "v", "dout") else torch.float32).contiguous()
            for k in keys + ("lam",)}
    B, H, T, dk, dv = w.B, w.H, w.T, w.dk, w.dv
    outs = {"dq": torch.empty((B, H, T, dk), dtype=td, device=dev), "dk": torch.empty((B, H, T, dk), dtype=td, device=dev),
            "dv": torch.empty((B, H, T, dv), dtype=td, device=dev),
            "dgamma": torch.empty((B, H, T), dtype=torch.float32, device=dev),
            "dlambda": torch.empty((H, dk), dtype=torch.float32, device=dev),
            "iters_fwd": torch.empty((B, H, T), dtype=torch.int32, device=dev),
            "iters_bwd": torch.empty((B, H, T), dtype=torch.int32, device=dev)}
    ws = torch.empty(binding.mesa_backward_workspace_size(B, H, T, dk, dv), dtype=torch.uint8, device=dev)
    _, _, xs = binding.mesa_forward_chunked_save(d_in["q"], d_in["k"], d_in["v"], d_in["gamma"], d_in["lam"],
                                                 w.cg_iters, w.cg_tol, w.chunk)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    in_bytes = sum(d_in[k].numel() * d_in[k].element_size() for k in keys)
    needs_flush = in_bytes < 2 * (129 << 20)

    def call(d, x_saved):
        binding.mesa_backward_chunked(d["q"], d["k"], d["v"], d["gamma"], d_in["lam"], d["dout"], w.cg_iters, w.cg_tol,
                                      workspace=ws, x_saved=x_saved, **outs)

    fl = (lambda: flush.random_(0, 255)) if needs_flush else None
    res = timed_loop(args, torch, lib, lambda i: call(d_in, xs), fl, world, dist, dev)
    res.update({"iters": outs["iters_bwd"].cpu().numpy(), "tokens_per_step": B * T, "flush": needs_flush})
    # the self-contained call (the forward's solves recomputed inside), a few steps
    rec = []
    for r in range(max(3, min(args.steps, 10)) + 1):
        if fl:
            fl()
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record()
        call(d_in, None)
        e_.record()
        torch.cuda.synchronize()
        if r:
            rec.append(s_.elapsed_time(e_))
    res["extra"] = {"x_saved": "from mesa_forward_chunked_save (untimed, before the loop)",
                    "ms_per_step_recomputing_the_forward_solves": float(np.median(rec))}
    if not args.no_e2e:
        h = {k: torch.from_numpy(inp[k]).to(td if k in ("q", "k", "v", "dout") else torch.float32).pin_memory()
             for k in keys}
        h["x_saved"] = xs.cpu().pin_memory()
        back = {k: torch.empty(outs[k].shape, dtype=outs[k].dtype).pin_memory() for k in ("dq", "dk", "dv", "dgamma", "dlambda")}

        bouts = [outs, {k: torch.empty_like(v) for k, v in outs.items()}]

        def run(d, stream, slot):
            binding.mesa_backward_chunked(d["q"], d["k"], d["v"], d["gamma"], d_in["lam"], d["dout"], w.cg_iters,
                                          w.cg_tol, workspace=ws, x_saved=d["x_saved"], stream=stream, **bouts[slot])
            return bouts[slot]

        ms = pipelined_e2e(torch, dev, h, run, back, max(3, min(args.steps, 20)))
        res["e2e"] = {"ms_per_step": ms, "h2d": sum(t.numel() * t.element_size() for t in h.values()),
                      "d2h": sum(t.numel() * t.element_size() for t in back.values())}
    return res


def aggregate(step_ms: float, tokens_per_rank: int, world: int, torch, dist, device="cuda"):
    """Whole-job figures of a replicated run: the slowest rank's time per step and the
    tokens of all ranks.  Each rank runs its own replica (independent sequences), so the
    only collective is this max."""
    if world > 1:
        t = torch.tensor([step_ms], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
    tokens = tokens_per_rank * world
    return step_ms, tokens, tokens / (step_ms / 1e3)


def emit(args, w, res, peaks, cpu, rank, world, torch, dist):
    step_ms, tokens, value = aggregate(float(np.sum(res["step_ms"])) / args.steps, res["tokens_per_step"],
                                       world, torch, dist)
    if rank != 0:
        return
    names = res["names"]
    kind_ms, kind_n = res["kind_ms"], res["kind_n"]
    top = int(np.argmax(kind_ms))
    top_name = names[top] if top < len(names) else f"kind{top}"
    launches = max(1, kind_n[top])
    avg_ms = kind_ms[top] / launches
    launches_per_step = sum(kind_n) / args.steps
    it = res["iters"]
    traffic = recorded_traffic(w.name, top_name)
    if w.conv_taps and not w.fused:
        bytes_ = preprocess_bytes(w)
        achieved = bytes_ / (avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "kernel": top_name,
                "peak_source": peaks["source"], "algorithmic_bytes": bytes_}
    elif w.decode_steps:
        bytes_ = decode_bytes(w)
        achieved = bytes_ / (avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "kernel": top_name,
                "peak_source": peaks["source"], "algorithmic_bytes": bytes_}
    else:
        if "cg" in top_name:
            # a backward solve has no readout: iterations only
            flops = cg_flops(w, it) - (0.0 if not w.backward else
                                       float(it.size) * (2.0 * w.dk * w.dk + 2.0 * w.dk * (w.chunk + 1)))
        elif "bwd_grad" in top_name:
            apart = any(n == "mesa_bwd_sprod_tc_kernel" and kind_n[i] > 0 for i, n in enumerate(names))
            flops = bwd_grad_flops(w, apart)
        elif "bwd_sprod" in top_name:
            flops = bwd_sprod_flops(w)
        elif "bwd_rhs" in top_name:
            flops = bwd_rhs_flops(w)
        else:
            flops = state_flops(w)
        achieved = flops / (avg_ms / 1e3) / 1e12
        if "_tc_" in top_name or "_tc64_" in top_name:
            # fp16 tcgen05 MMAs run at the bf16 dense rate; the measured cuBLAS bf16 peak
            peak = peaks["bf16_tflops"]
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic, "kernel": top_name,
                    "peak_source": f"{peaks['source']} bf16 dense (fp16 kind, same rate)",
                    "executed_tensor_tflops": (bwd_sprod_executed_flops(w) if "bwd_sprod" in top_name else
                                               tc_executed_flops(w, it, not w.backward)) / (avg_ms / 1e3) / 1e12}
        else:
            sms = peaks["sm_count"]
            peak = sms * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
            roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic, "kernel": top_name,
                    "peak_source": f"fp32 FMA: {sms} SMs (device) x 128 lanes x 2 flop x max SM clock"}
    kernels = {names[i] if i < len(names) else f"kind{i}": {"ms_per_step": kind_ms[i] / args.steps,
                                                             "launches": kind_n[i]}
               for i in range(len(kind_ms)) if kind_n[i] > 0}
    extra = {} if (w.conv_taps and not w.fused) else {"mean_iters": float(it.mean()), "max_iters": int(it.max())}
    extra["sm_count"] = peaks["sm_count"]
    extra["arithmetic"] = arithmetic(w)
    extra.update(res.get("extra", {}))
    extra.update({
             "l2": ("flushed between timed steps (256 MiB device write)" if res["flush"]
                    else "working set larger than L2, not flushed"),
             "kernels": kernels, "wall_s_timed_loop": res["wall_s"]})
    line = {"metric": METRIC_BWD if w.backward else METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded, see mesa_layer_gb300/synth.py)",
            "config": workload_config(w, extra), "roofline": roof, "cpu_baseline": cpu,
            "gpu_launches": int(sum(kind_n)), "launches_per_step": launches_per_step,
            "clocks": res["clocks"]}
    if "e2e" in res:
        e = res["e2e"]
        line["e2e"] = {"value": tokens / (e["ms_per_step"] / 1e3), "unit": "tokens/s",
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "ms_per_step": e["ms_per_step"]}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
