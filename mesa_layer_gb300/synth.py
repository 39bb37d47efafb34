"""Seeded synthetic inputs for the Mesa layer workloads.

This module only draws random numbers and shapes them into the input distributions of the
workloads; it holds none of the layer's arithmetic.  Both the CUDA path's tests and
benchmark and the CPU oracle take their inputs from here.

Recipe (every workload, seed 0 unless stated):
  * one independent numpy PCG64 stream per tensor, seeded with
    SeedSequence([seed, workload_id, tensor_id(, step)]);
  * q, k ~ N(0, 1) per element, then L2-normalised per token in fp64 (the pages put a
    normalisation of queries and keys before the layer);  v ~ N(0, 1);
  * gamma: U(lo, hi) or sigmoid(N(mu, sd)) as the workload states;
  * Lambda = diag(lambda), lambda ~ U(lo, hi), one vector per head;
  * every tensor is then rounded to the dtype the kernels read (fp32, or bf16 with
    round-to-nearest-even for q/k/v), and handed out as float32 arrays holding exactly
    those values, so the oracle sees what the GPU sees, upcast to fp64.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "gamma": 4, "lam": 5, "q_raw": 6, "k_raw": 7, "wq": 8, "wk": 9,
               "dout": 10}


@dataclass(frozen=True)
class Workload:
    name: str
    wid: int
    dtype: str                 # "f32" or "bf16" (q/k/v/out); gamma/lambda/states are fp32
    B: int
    H: int
    T: int
    dk: int
    dv: int
    chunk: int
    cg_iters: int              # fixed count if cg_tol <= 0, else the cap
    cg_tol: float
    gamma_kind: str            # "uniform" or "sigmoid"
    gamma_a: float
    gamma_b: float
    lam_lo: float
    lam_hi: float
    decode_steps: int = 0      # > 0: recurrent decode workload (B = sequences)
    prefix: int = 0            # decode: tokens folded into the state before the steps
    conv_taps: int = 0         # > 0: query/key preprocessing workload with this window
    warm: bool = False         # decode: each step's CG starts from the previous solution
    backward: bool = False     # the backward pass (gradients given dL/dout)
    fused: bool = False        # with conv_taps: the preprocessing fused into the forward

    @property
    def tokens(self) -> int:
        return self.B * self.T

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.T


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32_d16", 1, "f32", 1, 1, 256, 16, 16, 64, 16, 0.0,
                 "uniform", 0.90, 1.0, 0.25, 1.0),
        Workload("fwd_fp32_d64", 2, "f32", 2, 4, 2048, 64, 64, 64, 32, 1e-4,
                 "sigmoid", 3.0, 1.0, 0.1, 1.0),
        Workload("fwd_bf16_d128", 3, "bf16", 8, 16, 4096, 128, 128, 64, 15, 0.0,
                 "sigmoid", 4.0, 1.0, 0.05, 0.5),
        Workload("long_bf16_d128", 4, "bf16", 1, 16, 65536, 128, 128, 128, 30, 1e-3,
                 "sigmoid", 5.0, 1.5, 0.05, 0.5),
        Workload("decode_bf16_d128", 5, "bf16", 256, 16, 1, 128, 128, 64, 30, 1e-3,
                 "sigmoid", 4.0, 1.0, 0.05, 0.5, decode_steps=512, prefix=1024),
        # query/key preprocessing in front of the layer, on the shape of fwd_bf16_d128
        Workload("qkpre_bf16_d128", 6, "bf16", 8, 16, 4096, 128, 128, 64, 0, 0.0,
                 "sigmoid", 4.0, 1.0, 0.05, 0.5, conv_taps=4),
        # the decode workload with warm-started CG (inputs drawn as for decode_bf16_d128)
        Workload("decode_warm_bf16_d128", 5, "bf16", 256, 16, 1, 128, 128, 64, 30, 1e-3,
                 "sigmoid", 4.0, 1.0, 0.05, 0.5, decode_steps=512, prefix=1024, warm=True),
        # the backward pass on the shape and distributions of fwd_bf16_d128
        Workload("bwd_bf16_d128", 7, "bf16", 8, 16, 4096, 128, 128, 64, 15, 0.0,
                 "sigmoid", 4.0, 1.0, 0.05, 0.5, backward=True),
        # the forward of fwd_bf16_d128 on raw queries and keys, with the query/key
        # preprocessing (window 4) fused into it
        Workload("fwd_pre_bf16_d128", 8, "bf16", 8, 16, 4096, 128, 128, 64, 15, 0.0,
                 "sigmoid", 4.0, 1.0, 0.05, 0.5, conv_taps=4, fused=True),
    ]
}
WORKLOAD_ORDER = [w.name for w in sorted(WORKLOADS.values(), key=lambda w: w.wid)]


def workload(name_or_index, **overrides) -> Workload:
    """Look a workload up by name or by 1-based position, optionally shrunk."""
    if isinstance(name_or_index, int):
        w = WORKLOADS[WORKLOAD_ORDER[name_or_index - 1]]
    else:
        w = WORKLOADS[name_or_index]
    return replace(w, **overrides) if overrides else w


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _rng(seed: int, wid: int, tensor: str, step: int | None = None):
    key = [seed, wid, _TENSOR_IDS[tensor]] + ([] if step is None else [step + 1])
    return np.random.default_rng(np.random.SeedSequence(key))


def _unit_rows(rng, shape) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32).astype(np.float64)
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    n[n == 0] = 1.0
    return (x / n).astype(np.float32)


def _gamma(w: Workload, rng, shape) -> np.ndarray:
    if w.gamma_kind == "uniform":
        g = rng.uniform(w.gamma_a, w.gamma_b, size=shape)
    else:
        z = rng.normal(w.gamma_a, w.gamma_b, size=shape)
        g = 1.0 / (1.0 + np.exp(-z))
    return g.astype(np.float32)


def _cast(w: Workload, x: np.ndarray) -> np.ndarray:
    return round_bf16(x) if w.dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def lambdas(w: Workload, seed: int = 0) -> np.ndarray:
    """Lambda diagonal, [H, dk] float32."""
    return _rng(seed, w.wid, "lam").uniform(w.lam_lo, w.lam_hi, size=(w.H, w.dk)).astype(np.float32)


def forward_inputs(w: Workload, seed: int = 0) -> dict:
    """q, k [B, H, T, dk], v [B, H, T, dv], gamma [B, H, T], lam [H, dk] (float32 arrays,
    q/k/v already rounded to the workload dtype)."""
    B, H, T = w.B, w.H, w.T
    return {
        "q": _cast(w, _unit_rows(_rng(seed, w.wid, "q"), (B, H, T, w.dk))),
        "k": _cast(w, _unit_rows(_rng(seed, w.wid, "k"), (B, H, T, w.dk))),
        "v": _cast(w, _rng(seed, w.wid, "v").standard_normal(size=(B, H, T, w.dv), dtype=np.float32)),
        "gamma": _gamma(w, _rng(seed, w.wid, "gamma"), (B, H, T)),
        "lam": lambdas(w, seed),
    }


def backward_inputs(w: Workload, seed: int = 0) -> dict:
    """forward_inputs plus dout [B, H, T, dv] ~ N(0, 1) (the incoming gradient dL/dout),
    rounded to the workload dtype."""
    inp = forward_inputs(w, seed)
    shape = (w.B, w.H, w.T, w.dv)
    inp["dout"] = _cast(w, _rng(seed, w.wid, "dout").standard_normal(size=shape, dtype=np.float32))
    return inp


def decode_inputs(w: Workload, step: int, seed: int = 0) -> dict:
    """Inputs of one decode step (step < 0 for prefix tokens: step = -prefix .. -1):
    q, k [N, H, dk], v [N, H, dv], gamma [N, H]."""
    N, H = w.B, w.H
    s = step + w.prefix  # non-negative stream index
    return {
        "q": _cast(w, _unit_rows(_rng(seed, w.wid, "q", s), (N, H, w.dk))),
        "k": _cast(w, _unit_rows(_rng(seed, w.wid, "k", s), (N, H, w.dk))),
        "v": _cast(w, _rng(seed, w.wid, "v", s).standard_normal(size=(N, H, w.dv), dtype=np.float32)),
        "gamma": _gamma(w, _rng(seed, w.wid, "gamma", s), (N, H)),
    }


def preprocess_inputs(w: Workload, taps: int | None = None, seed: int = 0) -> dict:
    """Raw queries and keys of the preprocessing workloads: q_raw, k_raw [B, H, T, dk]
    ~ N(0, 1) rounded to the workload dtype; convolution taps wq, wk [H, dk, taps]
    ~ N(0, 1 / taps) in fp32 (tap s multiplies the input s tokens back)."""
    W = taps or w.conv_taps or 4
    shape = (w.B, w.H, w.T, w.dk)
    return {
        "q_raw": _cast(w, _rng(seed, w.wid, "q_raw").standard_normal(size=shape, dtype=np.float32)),
        "k_raw": _cast(w, _rng(seed, w.wid, "k_raw").standard_normal(size=shape, dtype=np.float32)),
        "wq": (_rng(seed, w.wid, "wq").standard_normal(size=(w.H, w.dk, W)) / np.sqrt(W)).astype(np.float32),
        "wk": (_rng(seed, w.wid, "wk").standard_normal(size=(w.H, w.dk, W)) / np.sqrt(W)).astype(np.float32),
    }
