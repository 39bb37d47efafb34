"""What fp32 arithmetic can reach on the fp32 workloads (CPU only).

A plain per-token restatement of the Mesa layer in numpy, with every operation in one chosen
floating-point type: the recurrence H_t = gamma_t H_{t-1} + k_t k_t^T, G_t likewise with
v_t k_t^T, textbook CG on (H_t + Lambda) x = q_t for a given number of iterations, and the
readout o_t = G_t x (MesaNet technical summary, gist.science/pt/paper/2506.05233, "A Camada
Mesa").  In float64 it reproduces the oracle (pinned below); in float32 it shows how far any
fp32 implementation of the same CG must expect to land from the fp64 oracle.

The finding that sets the GPU tests' metric for fp32 inputs: with the oracle's own iteration
counts, the fp32 restatement's per-token strict error ||o - o_ref|| / ||o_ref|| exceeds 1e-4
on the dynamic fp32 workload, always on tokens whose readout cancels (||o_t|| a few percent of
|| |G_t| |x_t| ||), while its error measured on the readout's magnitude stays well inside 1e-4.
The rounding that matters is that of the CG's matrix-vector products: the CG iterate moves by
~600 times the fp32 unit roundoff, and the cancelling readout magnifies that relative to
||o_t||.  These tests are the committed evidence; the numbers are quoted in the design notes.
"""
import numpy as np
import pytest

from helpers import oracle_forward, product_err, token_err
from mesa_layer_gb300 import synth


def restated_forward(inp, counts, dtype=np.float32, tol=0.0, counts_out=None):
    """o [B, H, T, dv] of the per-token recurrence and CG with every operation in `dtype`,
    token t running exactly counts[b, h, t] iterations (the batch axis is vectorised); with
    tol > 0 each token also stops before an iteration once ||r|| <= tol ||q|| (the stopping
    rule, evaluated in `dtype`), and counts_out [B, H, T] receives the iterations run."""
    q, k, v, g, lam = (inp[x] for x in ("q", "k", "v", "gamma", "lam"))
    B, H, T, d = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, H, T, dv))
    one, zero = dtype(1), dtype(0)
    for h in range(H):
        Hs = np.zeros((B, d, d), dtype)
        Gs = np.zeros((B, dv, d), dtype)
        L = lam[h].astype(dtype)
        for t in range(T):
            gt = g[:, h, t].astype(dtype)[:, None, None]
            kt, vt = k[:, h, t].astype(dtype), v[:, h, t].astype(dtype)
            Hs = gt * Hs + kt[:, :, None] * kt[:, None, :]
            Gs = gt * Gs + vt[:, :, None] * kt[:, None, :]
            x = np.zeros((B, d), dtype)
            r = q[:, h, t].astype(dtype)
            p = r.copy()
            rho = np.einsum("bi,bi->b", r, r)
            nq = np.sqrt(rho)
            n = counts[:, h, t]
            ran = np.zeros(B, dtype=np.int64)
            for it in range(int(n.max(initial=0))):
                act = it < n
                if tol > 0:
                    act = act & ~(np.sqrt(rho) <= dtype(tol) * nq)
                    n = np.where(act, n, np.minimum(n, it))
                ran += act
                w = np.einsum("bij,bj->bi", Hs, p) + L * p
                sig = np.einsum("bi,bi->b", p, w)
                ok = act & (sig > zero) & (rho > zero)
                al = np.where(ok, rho / np.where(sig > zero, sig, one), zero).astype(dtype)
                x = x + al[:, None] * p
                r = r - al[:, None] * w
                rn = np.einsum("bi,bi->b", r, r)
                be = np.where(act & (rho > zero), rn / np.where(rho > zero, rho, one), zero).astype(dtype)
                p = np.where(act[:, None], r + be[:, None] * p, p)
                rho = np.where(act, rn, rho)
            out[:, h, t] = np.einsum("bij,bj->bi", Gs, x)
            if counts_out is not None:
                counts_out[:, h, t] = ran
    return out


def test_restatement_is_the_oracle_in_fp64():
    """Pin: in float64 the restatement is the oracle (same recurrence, CG and counts), in
    fixed and in dynamic mode (8 iterations, and a stop at 1e-3, keep the fp64 rounding
    differences of the two summation orders far below the bound)."""
    for iters, tol in ((8, 0.0), (32, 1e-3)):
        w = synth.workload("fwd_fp32_d64", B=2, H=2, T=96, dk=32, dv=32, cg_iters=iters, cg_tol=tol)
        inp = synth.forward_inputs(w, seed=2)
        ro, rit, _ = oracle_forward(inp, w.cg_iters, w.cg_tol)
        o = restated_forward(inp, rit, np.float64)
        assert np.abs(o - ro).max() <= 1e-9 * np.abs(ro).max()


def _errors(inp, iters, tol):
    ro, rit, rs = oracle_forward(inp, iters, tol)
    o = restated_forward(inp, rit, np.float32)
    return token_err(o, ro), product_err(o, ro, rs)


def test_fp32_misses_strict_per_token_on_the_dynamic_workload():
    """The dynamic fp32 workload (d = 64, tol 1e-4, at most 32 iterations; its first batch
    row, four 2048-token sequences): fp32 exceeds 1e-4 per token on cancelling readouts and
    stays inside it on the readout's magnitude."""
    w = synth.workload("fwd_fp32_d64")
    inp = {k: (v[:1] if k != "lam" else v) for k, v in synth.forward_inputs(w).items()}
    strict, prod = _errors(inp, w.cg_iters, w.cg_tol)
    print(f"fp32 restatement, dynamic workload: strict max {strict.max():.3e}, tokens over 1e-4 "
          f"{int((strict > 1e-4).sum())} of {strict.size}, product-scale max {prod.max():.3e}")
    assert strict.max() > 3e-4
    assert prod.max() < 5e-5


@pytest.mark.parametrize("regime", ["gamma_near_zero", "gamma_one", "lambda_large", "zero_queries", "plain"])
def test_fp32_edge_regimes_unconverged(regime):
    """The GPU tests' edge regimes at 12 iterations (d = 32, not converged): fp32 on the
    readout's magnitude stays inside 1e-4 (closest: gates near zero, 8.0e-5, where every
    state is nearly the current token's rank-one term and a token's readout v_t (k_t . x)
    cancels in k_t . x; 8e-6 or less in the other regimes)."""
    w = synth.workload("fwd_fp32_d64", B=1, H=2, T=192, dk=32, dv=32, chunk=64, cg_iters=12, cg_tol=0.0)
    inp = synth.forward_inputs(w, seed=9)
    if regime == "gamma_near_zero":
        inp["gamma"][:] = np.float32(1e-3)
        inp["gamma"][0, 0, 70] = 0.0
    elif regime == "gamma_one":
        inp["gamma"][:] = 1.0
        inp["lam"][:] = 1.0
    elif regime == "lambda_large":
        inp["lam"][:] = 50.0
    elif regime == "zero_queries":
        inp["q"][0, 1, ::3] = 0.0
    strict, prod = _errors(inp, w.cg_iters, 0.0)
    print(f"fp32 restatement, {regime}: strict max {strict.max():.3e}, product-scale max {prod.max():.3e}")
    assert prod.max() < (1e-4 if regime == "gamma_near_zero" else 2.5e-5)


def test_fp32_chunk_invariance_case():
    """The chunk-invariance case of the GPU tests (d = 64, 16 fixed iterations)."""
    w = synth.workload("fwd_fp32_d64", B=1, H=2, T=256, dk=64, dv=64, cg_iters=16, cg_tol=0.0)
    inp = synth.forward_inputs(w, seed=3)
    strict, prod = _errors(inp, w.cg_iters, 0.0)
    print(f"fp32 restatement, d = 64 x 16 iterations: strict max {strict.max():.3e}, "
          f"product-scale max {prod.max():.3e}")
    assert prod.max() < 2.5e-5


def _near_zero_gates_d128(tol):
    """The tensor-core edge case of the GPU tests: bf16 inputs, d = 128, gates near zero."""
    w = synth.workload("fwd_bf16_d128", B=1, H=2, T=400, cg_iters=12 if tol == 0.0 else 30, cg_tol=tol)
    inp = synth.forward_inputs(w, seed=14)
    inp["gamma"][:] = np.float32(1e-3)
    inp["gamma"][0, 0, 170] = 0.0
    return w, inp


def test_fp32_near_zero_gates_d128_fixed():
    """Gates near zero at d = 128 (bf16 inputs, 12 un-converged iterations): every state is
    nearly the current token's rank-one term, the readout v_t (k_t . x) cancels in k_t . x, and
    fp32 arithmetic misses even the bf16 bound 2e-2 per token while its error on the readout's
    magnitude stays small.  The GPU test of this regime therefore asserts the latter."""
    w, inp = _near_zero_gates_d128(0.0)
    strict, prod = _errors(inp, w.cg_iters, 0.0)
    print(f"fp32 restatement, d = 128 gates near zero: strict max {strict.max():.3e}, "
          f"tokens over 2e-2 {int((strict > 2e-2).sum())} of {strict.size}, product-scale max {prod.max():.3e}")
    assert strict.max() > 2e-2
    assert prod.max() < 1e-3


def test_fp32_near_zero_gates_d128_dynamic_counts():
    """The same regime in dynamic mode (tol 1e-3): the fp32 restatement's own stopping
    decisions agree with the fp64 oracle's on fewer than half of the tokens (24 %, at most two
    iterations apart), so the GPU test of this regime checks every token against the oracle
    replaying the GPU's counts and does not hold the agreement rate to the usual floor."""
    w, inp = _near_zero_gates_d128(1e-3)
    ro, rit, rs = oracle_forward(inp, w.cg_iters, w.cg_tol)
    cnt = np.zeros_like(rit)
    restated_forward(inp, np.full_like(rit, w.cg_iters), np.float32, tol=w.cg_tol, counts_out=cnt)
    agree = float((cnt == rit).mean())
    print(f"fp32 restatement, d = 128 gates near zero, dynamic: counts agree {agree:.4f}, "
          f"max difference {int(np.abs(cnt - rit).max())}")
    assert agree < 0.5 and np.abs(cnt - rit).max() <= 3
