"""GPU parity of the backward pass (mesa_backward_chunked through the C ABI) against the fp64
oracle's backward: every d, both dtypes, ragged chunks, sequences spanning several chunks of
both chunk lengths (32 for the CUDA-core kernels, 128 for the tensor-core solves), a zero
incoming gradient, closed gates, dynamic mode, and the benchmark's workload at full size on
sampled (batch, head) units.

Metric: per (batch, head) unit, max |grad_gpu - grad_ref| / max |grad_ref| for dq, dk, dv and
dgamma; per head for dlambda (summed over the batch).  Tolerances as the forward's: 1e-4 for
fp32 inputs, 2e-2 for bf16 inputs (whose gradients are rounded to bf16 on output)."""
import numpy as np
import pytest

import oracle
from mesa_layer_gb300 import synth
from helpers import TOL, unit_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


def _wl(dtype, **kw):
    """Small cases: fp32 inputs take the fp32 workload's distributions (its Lambda range; the
    bf16 workload's smaller Lambda makes 15 un-converged fp32 CG steps conditioning-limited
    above 1e-4, on the CPU in plain fp32 as on the GPU), bf16 inputs the backward workload's."""
    if dtype == "f32":
        return synth.workload("fwd_fp32_d64", cg_tol=0.0, **kw)
    return synth.workload("bwd_bf16_d128", **kw)


def _dev(inp, dtype):
    import torch
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    return {k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda().to(td if k in ("q", "k", "v", "dout")
                                                                        else torch.float32).contiguous()
            for k in ("q", "k", "v", "gamma", "lam", "dout")}


def _gpu(inp, dtype, iters, tol, x_saved=None):
    import torch

    from mesa_layer_gb300 import binding
    t = _dev(inp, dtype)
    B, H, T, dk = t["q"].shape
    ws = torch.empty(max(256, binding.mesa_backward_workspace_size(B, H, T, dk, dk)), dtype=torch.uint8,
                     device="cuda")
    itf = torch.full((B, H, T), -1, dtype=torch.int32, device="cuda")
    dq, dk_, dv, dg, dl, itf, itb = binding.mesa_backward_chunked(t["q"], t["k"], t["v"], t["gamma"], t["lam"],
                                                                 t["dout"], iters, tol, workspace=ws,
                                                                 iters_fwd=itf, x_saved=x_saved)
    torch.cuda.synchronize()
    assert binding.mesa_forward_status(ws) == 0, "a kernel reported a bounded-wait timeout"
    f = lambda x: x.float().cpu().numpy().astype(np.float64)
    return {"dq": f(dq), "dk": f(dk_), "dv": f(dv), "dgamma": f(dg), "dlam": f(dl),
            "iters_fwd": itf.cpu().numpy(), "iters_bwd": itb.cpu().numpy()}


def _errs(g, r, mask=None):
    """Per-quantity max over units of the unit metric (dgamma as a one-feature sequence)."""
    e = {k: float(unit_err(g[k], r[k], mask).max()) for k in ("dq", "dk", "dv")}
    e["dgamma"] = float(unit_err(g["dgamma"][..., None], r["dgamma"][..., None], mask).max())
    e["dlam"] = float((np.abs(g["dlam"] - r["dlam"]).max(axis=-1) / np.abs(r["dlam"]).max(axis=-1)).max())
    return e


def _check(g, r, dtype, label, mask=None, counts=True):
    e = _errs(g, r, mask)
    print(f"{label}: " + ", ".join(f"{k} {v:.2e}" for k, v in e.items()))
    if counts:
        assert np.array_equal(g["iters_fwd"], r["iters_fwd"]) and np.array_equal(g["iters_bwd"], r["iters_bwd"])
    for k, v in e.items():
        assert v <= TOL[dtype], f"{label}: {k} {v:.3e}"
    return e


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_against_oracle_fixed(dtype, d):
    """75 tokens: two full 32-token chunks and a ragged one (one ragged 128-token chunk)."""
    w = _wl(dtype, B=2, H=2, T=75, dk=d, dv=d)
    inp = synth.backward_inputs(w, seed=d)
    g = _gpu(inp, dtype, 6, 0.0)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], inp["dout"], 6)
    _check(g, r, dtype, f"bwd d={d} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_several_chunks_d128(dtype):
    """300 tokens at d = 128: three 128-token chunks (tensor-core solves for bf16) and ten
    32-token chunks, the workload's 15 iterations."""
    w = _wl(dtype, B=1, H=3, T=300, dk=128, dv=128)
    inp = synth.backward_inputs(w, seed=5)
    g = _gpu(inp, dtype, 15, 0.0)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], inp["dout"], 15)
    _check(g, r, dtype, f"bwd T=300 {dtype}")


def test_single_token_and_zero_gradient():
    # one token: H + Lambda is Lambda plus one rank-1 term, d distinct eigenvalues, so CG is
    # run to convergence (d steps); an unconverged fixed-count fp32 iterate of such a spread
    # spectrum is an ill-conditioned function of rounding (a reordered dot product moved it
    # from 6e-5 to 1.9e-4 of the unit's scale at 8 steps)
    w = _wl("f32", B=2, H=2, T=1, dk=32, dv=32)
    inp = synth.backward_inputs(w, seed=1)
    g = _gpu(inp, "f32", 32, 0.0)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], inp["dout"], 32)
    _check(g, r, "f32", "bwd T=1")
    assert np.all(g["dgamma"] == 0.0)  # no earlier state
    w = _wl("f32", B=1, H=2, T=40, dk=64, dv=64)
    inp = synth.backward_inputs(w, seed=2)
    inp["dout"][:] = 0.0
    g = _gpu(inp, "f32", 8, 1e-4)
    for k in ("dq", "dk", "dv", "dgamma", "dlam"):
        assert np.all(g[k] == 0.0), k
    assert np.all(g["iters_bwd"] == 0)


def test_closed_gates():
    """Gates of exactly 0 cut the sequence: the GPU gives them a zero gate gradient (the
    forward clamps the log-gate there); every other gradient matches the oracle."""
    w = _wl("f32", B=1, H=2, T=70, dk=32, dv=32)
    inp = synth.backward_inputs(w, seed=3)
    inp["gamma"][:, :, [5, 33, 64]] = 0.0
    g = _gpu(inp, "f32", 8, 0.0)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], inp["dout"], 8)
    open_gate = inp["gamma"] > 0
    _check(g, r, "f32", "bwd closed gates", mask=open_gate)
    assert np.all(g["dgamma"][~open_gate] == 0.0)


def test_closed_gates_tensor_cores():
    """The same at bf16, d = 128 (the tensor-core solves, state sweeps and row x state
    products), over several 32- and 128-token chunks with a closed gate inside and at the
    first token of a 32-token chunk."""
    w = _wl("bf16", B=1, H=2, T=200, dk=128, dv=128)
    inp = synth.backward_inputs(w, seed=4)
    inp["gamma"][:, :, [7, 64, 150]] = 0.0
    g = _gpu(inp, "bf16", 10, 0.0)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], inp["dout"], 10)
    open_gate = inp["gamma"] > 0
    _check(g, r, "bf16", "bwd closed gates, tensor cores", mask=open_gate)
    assert np.all(g["dgamma"][~open_gate] == 0.0)


def test_units_are_independent_tensor_cores():
    """New inputs for batch row 1 leave every gradient of batch row 0 unchanged, bit for bit
    (bf16, d = 128: the tensor-core solves with segment carries, the sweeps, the products)."""
    w = _wl("bf16", B=2, H=2, T=300, dk=128, dv=128)
    a = synth.backward_inputs(w, seed=8)
    b = synth.backward_inputs(w, seed=9)
    g = _gpu(a, "bf16", 10, 0.0)
    mixed = dict(a)
    for key in ("q", "k", "v", "gamma", "dout"):
        mixed[key] = a[key].copy()
        mixed[key][1] = b[key][1]
    g2 = _gpu(mixed, "bf16", 10, 0.0)
    for name in ("dq", "dk", "dv", "dgamma"):
        assert np.array_equal(g2[name][0], g[name][0]), name
        assert not np.array_equal(g2[name][1], g[name][1]), name


def test_gradient_scale_is_exact():
    """Every gradient is linear in dL/dout, and the tensor-core path (bf16, d = 128: the
    solves, the state sweeps, the row x state products) takes its operand scales from
    exponent bits: dout times 2^k (k = -30, 30) gives exactly 2^k times every gradient, bit
    for bit, with the same counts."""
    w = _wl("bf16", B=1, H=2, T=200, dk=128, dv=128)
    inp = synth.backward_inputs(w, seed=6)
    g = _gpu(inp, "bf16", 10, 0.0)
    for k in (-30, 30):
        sc = dict(inp)
        sc["dout"] = (inp["dout"] * 2.0 ** k).astype(inp["dout"].dtype)
        g2 = _gpu(sc, "bf16", 10, 0.0)
        assert np.array_equal(g2["iters_bwd"], g["iters_bwd"]), k
        for name in ("dq", "dk", "dv", "dgamma", "dlam"):
            assert np.array_equal(g2[name], g[name] * 2.0 ** k), (k, name)


def test_dynamic_mode():
    """Dynamic stopping (tol 1e-3, cap 30): counts may differ at the threshold; the units whose
    counts all agree must meet the tolerance, and at least 95 % of the counts agree."""
    w = _wl("f32", B=2, H=2, T=96, dk=64, dv=64)
    inp = synth.backward_inputs(w, seed=4)
    g = _gpu(inp, "f32", 30, 1e-3)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], inp["dout"], 30, 1e-3)
    agree = (g["iters_fwd"] == r["iters_fwd"]) & (g["iters_bwd"] == r["iters_bwd"])
    print(f"bwd dynamic: counts agree {agree.mean():.4f}, mean iters fwd {g['iters_fwd'].mean():.2f} "
          f"bwd {g['iters_bwd'].mean():.2f}")
    assert agree.mean() >= 0.95
    units = agree.all(axis=-1)
    for b, h in zip(*np.nonzero(units)):
        e = {k: float(unit_err(g[k][b, h], r[k][b, h])) for k in ("dq", "dk", "dv")}
        e["dgamma"] = float(unit_err(g["dgamma"][b, h][:, None], r["dgamma"][b, h][:, None]))
        for k, v in e.items():
            assert v <= TOL["f32"], f"unit ({b}, {h}) {k} {v:.3e}"


def test_full_workload_sampled_units():
    """The benchmark's backward workload (B=8 H=16 T=4096 d=128 bf16, 15 iterations), all
    units on the GPU; the oracle follows three (batch, head) units (dlambda, a sum over the
    batch, is covered by the small cases)."""
    w = synth.workload("bwd_bf16_d128")
    inp = synth.backward_inputs(w)
    g = _gpu(inp, w.dtype, w.cg_iters, w.cg_tol)
    assert np.all(g["iters_fwd"] == w.cg_iters) and np.all(g["iters_bwd"] == w.cg_iters)
    units = ((0, 0), (3, 7), (7, 15))
    bs, hs = [u[0] for u in units], [u[1] for u in units]
    # the sampled units side by side as three heads of one sequence batch (each its own lambda)
    sub = {k: inp[k][bs, hs][None] for k in ("q", "k", "v", "gamma", "dout")}
    r = oracle.backward(sub["q"], sub["k"], sub["v"], sub["gamma"], inp["lam"][hs], sub["dout"],
                        w.cg_iters, w.cg_tol)
    for n, (b, h) in enumerate(units):
        e = {k: float(unit_err(g[k][b, h], r[k][0, n])) for k in ("dq", "dk", "dv")}
        e["dgamma"] = float(unit_err(g["dgamma"][b, h][:, None], r["dgamma"][0, n][:, None]))
        print(f"bwd full b={b} h={h}: " + ", ".join(f"{k} {v:.2e}" for k, v in e.items()))
        for k, v in e.items():
            assert v <= TOL[w.dtype], f"({b}, {h}) {k} {v:.3e}"


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 128), ("f32", 64), ("bf16", 32)])
def test_saved_iterates(dtype, d):
    """mesa_forward_chunked_save gives the forward's outputs bit for bit plus its iterates;
    the backward from them matches the oracle (and, on the tensor-core path, where the
    recomputation runs the same kernel on the same chunks, the recomputing backward bit for
    bit); iters_fwd is then left alone."""
    import torch

    from mesa_layer_gb300 import binding
    w = _wl(dtype, B=2, H=2, T=150, dk=d, dv=d)
    inp = synth.backward_inputs(w, seed=9)
    t = _dev(inp, dtype)
    o0, i0 = binding.mesa_forward_chunked(t["q"], t["k"], t["v"], t["gamma"], t["lam"], 10, 0.0, w.chunk)
    o1, i1, xs = binding.mesa_forward_chunked_save(t["q"], t["k"], t["v"], t["gamma"], t["lam"], 10, 0.0, w.chunk)
    assert torch.equal(o0, o1) and torch.equal(i0, i1)
    g1 = _gpu(inp, dtype, 10, 0.0, x_saved=xs)
    assert np.all(g1["iters_fwd"] == -1)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], inp["dout"], 10)
    g1["iters_fwd"] = r["iters_fwd"]
    _check(g1, r, dtype, f"bwd saved iterates d={d} {dtype}")
    if dtype == "bf16" and d == 128:
        g0 = _gpu(inp, dtype, 10, 0.0)
        for k in ("dq", "dk", "dv", "dgamma", "dlam"):
            assert np.array_equal(g0[k], g1[k]), k


def test_dynamic_mode_tensor_cores():
    """Dynamic stopping on the tensor-core path (bf16, d = 128, tol 1e-3, cap 30, the long
    workload's rule): both solves stop per token; at least 95 % of the counts agree with the
    oracle's and the units whose counts all agree meet the bf16 tolerance."""
    w = synth.workload("bwd_bf16_d128", B=2, H=2, T=256, cg_iters=30, cg_tol=1e-3)
    inp = synth.backward_inputs(w, seed=6)
    g = _gpu(inp, "bf16", 30, 1e-3)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], inp["dout"], 30, 1e-3)
    agree = (g["iters_fwd"] == r["iters_fwd"]) & (g["iters_bwd"] == r["iters_bwd"])
    print(f"bwd dynamic tc: counts agree {agree.mean():.4f}, mean iters fwd {g['iters_fwd'].mean():.2f} "
          f"bwd {g['iters_bwd'].mean():.2f}")
    assert agree.mean() >= 0.95
    for b, h in zip(*np.nonzero(agree.all(axis=-1))):
        e = {k: float(unit_err(g[k][b, h], r[k][b, h])) for k in ("dq", "dk", "dv")}
        e["dgamma"] = float(unit_err(g["dgamma"][b, h][:, None], r["dgamma"][b, h][:, None]))
        for k, v in e.items():
            assert v <= TOL["bf16"], f"unit ({b}, {h}) {k} {v:.3e}"
