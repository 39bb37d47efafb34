"""Tensor-core building blocks (tcgen05.mma with the swizzled fp16 operand layouts the
chunked CG uses) against a plain matrix product, and the tensor-core forward path against
the oracle on shapes that exercise its tiling."""
import numpy as np
import pytest

import oracle
from mesa_layer_gb300 import synth
from helpers import forward_check, gpu_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


def test_tc_selftest_matches_fp16_products():
    import torch

    from mesa_layer_gb300 import binding
    rng = np.random.default_rng(0)
    A = rng.standard_normal((128, 128)).astype(np.float32)
    B = rng.standard_normal((128, 128)).astype(np.float32)
    A[3, :] = 0.0
    B[:, 7] *= 1e-3
    C1, C2, C3, st = binding.mesa_tc_selftest(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    a16 = A.astype(np.float16).astype(np.float64)
    b16 = B.astype(np.float16).astype(np.float64)
    np.testing.assert_allclose(C1.cpu().numpy(), a16 @ b16.T, rtol=1e-5, atol=1e-4)
    np.testing.assert_allclose(C2.cpu().numpy(), a16 @ b16, rtol=1e-5, atol=1e-4)
    np.testing.assert_allclose(C3.cpu().numpy(), a16.T @ b16, rtol=1e-5, atol=1e-4)


TC_CASES = [
    # (B, H, T, iters, tol, note)
    (1, 1, 128, 8, 0.0, "one full chunk"),
    (1, 2, 300, 15, 0.0, "ragged last chunk"),
    (2, 1, 520, 30, 1e-3, "dynamic"),
    (1, 1, 96, 0, 0.0, "zero iterations"),
    (1, 3, 1000, 30, 1e-3, "dynamic several chunks"),
    (2, 1, 640, 30, 1e-4, "dynamic tight tolerance"),
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: c[-1].replace(" ", "_"))
def test_tc_forward_against_oracle(case):
    B, H, T, iters, tol, _ = case
    w = synth.workload("fwd_bf16_d128", B=B, H=H, T=T, cg_iters=iters, cg_tol=tol)
    inp = synth.forward_inputs(w, seed=11)
    o, it = gpu_forward(inp, "bf16", iters, tol, 64)
    r = forward_check(inp, o, it, "bf16", iters, tol, case[-1])
    print(f"tc {case[-1]}: {r}")
    if iters == 0:
        assert np.all(o == 0)


def test_tc_initial_state_and_final_states():
    import torch

    w = synth.workload("fwd_bf16_d128", B=1, H=2, T=384, cg_iters=12, cg_tol=0.0)
    inp = synth.forward_inputs(w, seed=12)
    _, _, Hf, Gf = oracle.forward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], 0, 0.0,
                                  want_final=True)
    t1 = 200
    first = {k: (v[:, :, :t1] if k != "lam" else v) for k, v in inp.items()}
    second = {k: (v[:, :, t1:] if k != "lam" else v) for k, v in inp.items()}
    H1 = torch.empty(1, 2, 128, 128, device="cuda")
    G1 = torch.empty_like(H1)
    Hg, Gg = torch.empty_like(H1), torch.empty_like(H1)
    o1, i1 = gpu_forward(first, "bf16", 12, 0.0, 64, H_final=H1, G_final=G1)
    o2, i2 = gpu_forward(second, "bf16", 12, 0.0, 64, H0=H1, G0=G1, H_final=Hg, G_final=Gg)
    o = np.concatenate([o1, o2], axis=2)
    forward_check(inp, o, np.concatenate([i1, i2], axis=2), "bf16", 12, 0.0, "split")
    for a, b in ((Hg, Hf), (Gg, Gf)):
        a = a.cpu().numpy().astype(np.float64)
        assert np.abs(a - b).max() <= 1e-5 * np.abs(b).max()


def test_tc_many_segments_with_initial_state():
    """A single long sequence (40 chunks): the state build splits it into segments that start
    from zero and are chained by carries; outputs and final states must not notice."""
    import torch

    w = synth.workload("fwd_bf16_d128", B=1, H=1, T=40 * 128 - 17, cg_iters=10, cg_tol=0.0)
    inp = synth.forward_inputs(w, seed=13)
    rng = np.random.default_rng(13)
    M = rng.standard_normal((1, 1, 128, 128)).astype(np.float32) * 0.1
    H0 = (M @ np.swapaxes(M, -1, -2)).astype(np.float32)       # symmetric PSD start state
    G0 = (rng.standard_normal((1, 1, 128, 128)) * 0.1).astype(np.float32)
    _, _, Hf, Gf = oracle.forward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], 0, 0.0,
                                  H0=H0, G0=G0, want_final=True)
    Hg = torch.empty(1, 1, 128, 128, device="cuda")
    Gg = torch.empty_like(Hg)
    o, it = gpu_forward(inp, "bf16", 10, 0.0, 128, H0=torch.from_numpy(H0).cuda(),
                        G0=torch.from_numpy(G0).cuda(), H_final=Hg, G_final=Gg)
    r = forward_check(inp, o, it, "bf16", 10, 0.0, "segments", H0=H0, G0=G0)
    for a, b in ((Hg, Hf), (Gg, Gf)):
        a = a.cpu().numpy().astype(np.float64)
        assert np.abs(a - b).max() <= 1e-5 * np.abs(b).max()
    print(f"tc segments: {r}")


@pytest.mark.parametrize("tol", [0.0, 1e-3], ids=["fixed", "dynamic"])
@pytest.mark.parametrize("regime", ["gamma_near_zero", "gamma_one", "lambda_large", "zero_queries"])
def test_tc_edge_values(regime, tol):
    """The edge regimes on the tensor-core path (bf16, d = 128, three chunks and a ragged
    tail), fixed at 12 un-converged iterations and dynamic, every token against the oracle."""
    w = synth.workload("fwd_bf16_d128", B=1, H=2, T=400, cg_iters=12 if tol == 0.0 else 30, cg_tol=tol)
    inp = synth.forward_inputs(w, seed=14)
    if regime == "gamma_near_zero":
        inp["gamma"][:] = np.float32(1e-3)
        inp["gamma"][0, 0, 170] = 0.0
    elif regime == "gamma_one":
        inp["gamma"][:] = 1.0
        inp["lam"][:] = 1.0
    elif regime == "lambda_large":
        inp["lam"][:] = 50.0
    else:
        inp["q"][0, 1, ::3] = 0.0
    o, it = gpu_forward(inp, "bf16", w.cg_iters, tol, 64)
    kw = {}
    if regime == "gamma_near_zero":
        # every state is nearly the current token's rank-one term and the readout v_t (k_t . x)
        # cancels: a plain fp32 restatement misses 2e-2 per token there too (1.3 at worst) and
        # agrees with the fp64 stopping decisions on 24 % of the tokens (test_fp32_rounding.py),
        # so this regime is checked on the readout's magnitude, every token at the GPU's count
        kw = dict(metric="product", min_agree=0.1)
    r = forward_check(inp, o, it, "bf16", w.cg_iters, tol, f"tc {regime} tol {tol}", **kw)
    print(f"tc {regime} tol {tol}: {r}")
    if regime == "zero_queries":
        assert np.all(o[0, 1, ::3] == 0)
        if tol > 0:
            assert np.all(it[0, 1, ::3] == 0)


def test_tc_dynamic_initial_state():
    """Dynamic mode continued from a state (the first chunk then has a nonzero state too)."""
    import torch

    w = synth.workload("long_bf16_d128", B=1, H=2, T=700)
    inp = synth.forward_inputs(w, seed=15)
    rng = np.random.default_rng(15)
    M = rng.standard_normal((1, 2, 128, 128)).astype(np.float32) * 0.1
    H0 = (M @ np.swapaxes(M, -1, -2)).astype(np.float32)
    G0 = (rng.standard_normal((1, 2, 128, 128)) * 0.1).astype(np.float32)
    o, it = gpu_forward(inp, "bf16", w.cg_iters, w.cg_tol, 128, H0=torch.from_numpy(H0).cuda(),
                        G0=torch.from_numpy(G0).cuda())
    r = forward_check(inp, o, it, "bf16", w.cg_iters, w.cg_tol, "dynamic from a state", H0=H0, G0=G0)
    print(f"tc dynamic from a state: {r}")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_tc_units_are_independent(dtype, d):
    """A unit's outputs do not depend on any other unit's inputs: with B*H = 4 units of eight
    128-token chunks the state build runs one segment per chunk and the CG kernel adds the
    segment carries, so a wrong unit, chunk or segment index anywhere would mix units.  New
    inputs for batch row 1 leave batch row 0's outputs and counts unchanged, bit for bit."""
    w = synth.workload("fwd_bf16_d128" if dtype == "bf16" else "fwd_fp32_d64", dtype=dtype, dk=d, dv=d, B=2, H=2,
                       T=1000, cg_iters=30, cg_tol=1e-3)
    a = synth.forward_inputs(w, seed=23)
    b = synth.forward_inputs(w, seed=24)
    o, it = gpu_forward(a, dtype, w.cg_iters, w.cg_tol, 64)
    mixed = dict(a)
    for key in ("q", "k", "v", "gamma"):
        mixed[key] = a[key].copy()
        mixed[key][1] = b[key][1]
    o2, it2 = gpu_forward(mixed, dtype, w.cg_iters, w.cg_tol, 64)
    assert np.array_equal(o2[0], o[0]) and np.array_equal(it2[0], it[0])
    assert not np.array_equal(o2[1], o[1])


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
@pytest.mark.parametrize("tol", [0.0, 1e-3], ids=["fixed", "dynamic"])
def test_tc_value_scale_is_exact(dtype, d, tol):
    """The readout is linear in v and the CG does not see v: v times 2^k (k = -40, 40) gives
    exactly 2^k times the outputs with the same counts.  The value operands' scales come from
    exponent bits, so the products see the same fp16 operands at every k: a check of those
    scale paths over a wide range of exponents (the state build's and the readout's)."""
    w = synth.workload("fwd_bf16_d128" if dtype == "bf16" else "fwd_fp32_d64", dtype=dtype, dk=d, dv=d, B=1, H=2,
                       T=300, cg_iters=12 if tol == 0.0 else 30, cg_tol=tol)
    inp = synth.forward_inputs(w, seed=19)
    o, it = gpu_forward(inp, dtype, w.cg_iters, tol, 64)
    for k in (-40, 40):
        sc = dict(inp)
        sc["v"] = (inp["v"] * np.float32(2.0 ** k)).astype(np.float32)
        o2, it2 = gpu_forward(sc, dtype, w.cg_iters, tol, 64)
        assert np.array_equal(it2, it), k
        assert np.array_equal(o2, (o * np.float32(2.0 ** k)).astype(np.float32)), k


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
@pytest.mark.parametrize("tol", [0.0, 1e-3], ids=["fixed", "dynamic"])
def test_tc_query_scale_is_exact(dtype, d, tol):
    """The CG iterate is homogeneous in q, and the tensor-core kernels take every operand scale
    from exponent bits: q times 2^k (k = -40, 40) gives exactly 2^k times the outputs, bit for
    bit, with the same iteration counts (the stopping rule compares norms that scale alike),
    and the scaled call still matches the oracle -- on the readout's magnitude: at 12
    un-converged iterations one token of this case has a cancelling readout (strict 2.2e-2,
    as in the unscaled call, whose outputs are the same bits up to the power of two)."""
    w = synth.workload("fwd_bf16_d128" if dtype == "bf16" else "fwd_fp32_d64", dtype=dtype, dk=d, dv=d, B=1, H=2,
                       T=300, cg_iters=12 if tol == 0.0 else 30, cg_tol=tol)
    inp = synth.forward_inputs(w, seed=17)
    o, it = gpu_forward(inp, dtype, w.cg_iters, tol, 64)
    for k in (-40, 40):
        sc = dict(inp)
        sc["q"] = (inp["q"] * np.float32(2.0 ** k)).astype(np.float32)
        o2, it2 = gpu_forward(sc, dtype, w.cg_iters, tol, 64)
        assert np.array_equal(it2, it), k
        assert np.array_equal(o2, (o * np.float32(2.0 ** k)).astype(np.float32)), k
    r = forward_check(sc, o2, it2, dtype, w.cg_iters, tol, f"q x 2^{k}", metric="product")
    print(f"q x 2^{k}: {r}")
