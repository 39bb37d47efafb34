"""Shared helpers of the GPU parity tests: device upload, error metrics, oracle checks.

Acceptance metric (the reading of "max relative error"): for every independent unit (one
(batch, head) sequence, or one decode (sequence, head) over its steps) the largest absolute
output error divided by the largest absolute reference output of that unit,
    err_unit = max |o_gpu - o_ref| / max |o_ref|,
and the check takes the max over units.  The per-token ratio ||o_gpu,t - o_ref,t|| / ||o_ref,t||
is also reported (not asserted): when a token's output has cancelled to a small norm and CG
has not converged, fp32 and fp64 runs of the same CG differ by far more than fp32 rounding
(the un-converged iterate is an ill-conditioned function of the data), so that ratio measures
the problem's conditioning rather than the kernel.
"""
from __future__ import annotations

import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}


def unit_err(o_gpu, o_ref, mask=None) -> np.ndarray:
    """err per unit: arrays [..., tokens, features]; returns [...] (leading unit axes).
    mask [..., tokens] selects the tokens whose error counts (default: all)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    d = np.abs(o_gpu - o_ref)
    if mask is not None:
        d = np.where(mask[..., None], d, 0.0)
    scale = np.abs(o_ref).max(axis=(-1, -2))
    return d.max(axis=(-1, -2)) / np.maximum(scale, 1e-300)


def token_err(o_gpu, o_ref) -> np.ndarray:
    """Per-token ||o_gpu - o_ref|| / ||o_ref|| (reported only)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    return np.linalg.norm(o_gpu - o_ref, axis=-1) / np.maximum(np.linalg.norm(o_ref, axis=-1), 1e-300)


# kept for callers comparing two GPU results with each other
rel_err = unit_err


def torch_inputs(inp: dict, dtype: str, device="cuda"):
    import torch
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = {}
    for key in ("q", "k", "v"):
        out[key] = torch.from_numpy(np.ascontiguousarray(inp[key])).to(device=device, dtype=td).contiguous()
    for key in ("gamma", "lam"):
        out[key] = torch.from_numpy(np.ascontiguousarray(inp[key])).to(device=device, dtype=torch.float32).contiguous()
    return out


def gpu_forward(inp: dict, dtype: str, cg_iters: int, cg_tol: float, chunk: int, **kw):
    import torch

    from mesa_layer_gb300 import binding
    t = torch_inputs(inp, dtype)
    B, H, T, dk = t["q"].shape
    ws = torch.empty(max(256, binding.mesa_forward_workspace_size(B, H, T, dk, t["v"].shape[-1], chunk)),
                     dtype=torch.uint8, device="cuda")
    out, it = binding.mesa_forward_chunked(t["q"], t["k"], t["v"], t["gamma"], t["lam"], cg_iters,
                                           cg_tol, chunk, workspace=ws, **kw)
    torch.cuda.synchronize()
    if T > 0:
        assert binding.mesa_forward_status(ws) == 0, "a kernel reported a bounded-wait timeout"
    return out.float().cpu().numpy().astype(np.float64), it.cpu().numpy()


def check_against_oracle(o_gpu, it_gpu, o_ref, it_ref, dtype, dynamic, label="", min_agree=0.95):
    """Arrays are [..., tokens, features] / [..., tokens].  ``dynamic`` is the CG tolerance
    (0 for fixed mode).
    Fixed mode: identical iteration counts everywhere and err_unit within the dtype tolerance.
    Dynamic mode: the tokens whose counts agree must meet the tolerance; counts may differ
    by one or two for tokens at the stopping threshold (fp32 and fp64 residuals cross it at
    different iterations) on at most 1 - min_agree of the tokens, and those tokens, which
    meet the stopping rule on both sides, must lie within cg_tol times a condition-number
    allowance.  Returns (max err_unit, per-token errors)."""
    tol = TOL[dtype]
    tok = token_err(o_gpu, o_ref)
    if not dynamic:
        assert np.array_equal(it_gpu, it_ref), f"{label}: iteration counts differ"
        e = unit_err(o_gpu, o_ref)
        assert e.max() <= tol, f"{label}: max rel err {e.max():.3e} > {tol}"
        return e.max(), tok
    same = it_gpu == it_ref
    diff = np.abs(it_gpu.astype(np.int64) - it_ref)
    assert same.mean() >= min_agree, f"{label}: only {same.mean():.3f} of counts agree"
    assert diff.max() <= 2, f"{label}: count differs by {diff.max()}"
    e = unit_err(o_gpu, o_ref, same)
    assert e.max() <= tol, f"{label}: max rel err {e.max():.3e} > {tol}"
    if (~same).any():
        eo = unit_err(o_gpu, o_ref, ~same)
        assert eo.max() <= max(tol, 200 * dynamic), f"{label}: off-count tokens err {eo.max():.3e}"
    return e.max(), tok
