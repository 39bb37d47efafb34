"""GPU parity of the chunked forward (mesa_forward_chunked through the C ABI) against the
fp64 oracle, on the five workloads' forward configurations and on edge cases."""
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


def test_tiny_fp32_d16_full():
    """The tiny fp32 workload (d = 16, 16 iterations: CG has converged), strict per-token."""
    w = synth.workload("tiny_fp32_d16")
    inp = synth.forward_inputs(w)
    o, it = gpu_forward(inp, w.dtype, w.cg_iters, w.cg_tol, w.chunk)
    r = forward_check(inp, o, it, w.dtype, w.cg_iters, w.cg_tol, "tiny", metric="strict")
    assert (it == 16).all()
    print(f"tiny: {r}")


def test_fp32_d64_dynamic_full():
    """The dynamic fp32 workload at full size: every token against the oracle replaying the
    GPU's own counts, on the readout's magnitude (strict per-token reported)."""
    w = synth.workload("fwd_fp32_d64")
    inp = synth.forward_inputs(w)
    o, it = gpu_forward(inp, w.dtype, w.cg_iters, w.cg_tol, w.chunk)
    r = forward_check(inp, o, it, w.dtype, w.cg_iters, w.cg_tol, "fp32_d64")
    print(f"fp32_d64: {r}, mean iters {it.mean():.2f}")


def _unit_inputs(inp, b, h, t0=0, t1=None):
    """One (batch, head) unit over tokens [t0, t1) as a 1 x 1 batch, with its lambda row."""
    sl = {k: inp[k][b, h][None, None, t0:t1] for k in ("q", "k", "v", "gamma")}
    sl["lam"] = inp["lam"][h][None]
    return sl


def _check_units(w, inp, o, it, units, t0=0, t1=None, label=""):
    """Oracle on selected units over tokens [t0, t1); the state at t0 comes from the
    oracle's own state-only pass (cg_iters = 0) over tokens [0, t0)."""
    import oracle
    results = []
    for b, h in units:
        kw = {}
        if t0 > 0:
            pre = _unit_inputs(inp, b, h, 0, t0)
            _, _, H0, G0 = oracle.forward(pre["q"], pre["k"], pre["v"], pre["gamma"], pre["lam"], 0, 0.0,
                                          want_final=True)
            kw = {"H0": H0, "G0": G0}
        sub = _unit_inputs(inp, b, h, t0, t1)
        og = o[b, h, t0:t1][None, None]
        ig = it[b, h, t0:t1][None, None]
        results.append(forward_check(sub, og, ig, w.dtype, w.cg_iters, w.cg_tol, f"{label}({b},{h})[{t0}:{t1}]",
                                     **kw))
    return results


def test_bf16_d128_full_size_sampled_units():
    w = synth.workload("fwd_bf16_d128")
    inp = synth.forward_inputs(w)
    o, it = gpu_forward(inp, w.dtype, w.cg_iters, w.cg_tol, w.chunk)
    assert (it == w.cg_iters).all()
    for r in _check_units(w, inp, o, it, [(0, 0), (3, 7), (7, 15)], label="bf16_d128"):
        print(f"bf16_d128: {r}")


def test_long_bf16_full_size_sampled_windows():
    w = synth.workload("long_bf16_d128")
    inp = synth.forward_inputs(w)
    o, it = gpu_forward(inp, w.dtype, w.cg_iters, w.cg_tol, w.chunk)
    assert it.min() >= 0 and it.max() <= w.cg_iters
    for (b, h), (t0, t1) in [((0, 0), (0, 2048)), ((0, 11), (w.T - 2048, w.T))]:
        r, = _check_units(w, inp, o, it, [(b, h)], t0, t1, label="long")
        print(f"long head {h} tokens {t0}:{t1}: {r}")


EDGE = [
    # (dtype, B, H, T, d, chunk, iters, tol)
    ("f32", 1, 1, 1, 16, 16, 4, 0.0),          # a single token
    ("f32", 1, 2, 100, 32, 32, 12, 0.0),       # ragged last chunk
    ("f32", 2, 1, 130, 64, 64, 20, 1e-5),      # ragged, dynamic
    ("f32", 1, 1, 200, 128, 128, 10, 0.0),     # d = 128, ragged
    ("bf16", 1, 2, 257, 128, 64, 15, 0.0),     # bf16, several tiles and a 1-token tail
    ("bf16", 2, 2, 96, 64, 16, 8, 1e-3),       # small chunks, dynamic
    ("f32", 3, 1, 64, 16, 64, 0, 0.0),         # zero iterations: o = 0
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "-".join(map(str, c)))
def test_edge_shapes(case):
    dtype, B, H, T, d, chunk, iters, tol = case
    w = synth.workload("fwd_fp32_d64", dtype=dtype, B=B, H=H, T=T, dk=d, dv=d, chunk=chunk,
                       cg_iters=iters, cg_tol=tol)
    inp = synth.forward_inputs(w, seed=5)
    o, it = gpu_forward(inp, dtype, iters, tol, chunk)
    r = forward_check(inp, o, it, dtype, iters, tol, str(case))
    print(f"{case}: {r}")
    if iters == 0:
        assert np.all(o == 0)


@pytest.mark.parametrize("regime", ["gamma_near_zero", "gamma_one", "lambda_large", "zero_queries"])
def test_edge_values(regime):
    """Edge regimes at 12 iterations (d = 32: CG has not converged), every token."""
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
    else:
        inp["q"][0, 1, ::3] = 0.0
    o, it = gpu_forward(inp, w.dtype, w.cg_iters, w.cg_tol, w.chunk)
    r = forward_check(inp, o, it, w.dtype, w.cg_iters, 0.0, regime)
    print(f"{regime}: {r}")
    if regime == "zero_queries":
        assert np.all(o[0, 1, ::3] == 0)
        # dynamic mode stops zero queries before the first iteration
        o2, it2 = gpu_forward(inp, w.dtype, 48, 1e-3, w.chunk)
        assert np.all(it2[0, 1, ::3] == 0) and np.all(o2[0, 1, ::3] == 0)
        forward_check(inp, o2, it2, w.dtype, 48, 1e-3, "zero_queries dynamic")


def test_chunk_size_invariance():
    """d = 64, 16 iterations (not converged): every chunk length against the oracle, per token."""
    w = synth.workload("fwd_fp32_d64", B=1, H=2, T=256, dk=64, dv=64, cg_iters=16, cg_tol=0.0)
    inp = synth.forward_inputs(w, seed=3)
    for c in (16, 32, 64, 128):
        o, it = gpu_forward(inp, w.dtype, w.cg_iters, 0.0, c)
        r = forward_check(inp, o, it, w.dtype, w.cg_iters, 0.0, f"chunk {c}")
        print(f"chunk {c}: {r}")


def test_initial_and_final_states():
    import oracle
    import torch

    w = synth.workload("fwd_fp32_d64", B=2, H=2, T=160, cg_iters=10, cg_tol=0.0)
    inp = synth.forward_inputs(w, seed=4)
    _, _, Hf, Gf = oracle.forward(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["lam"], 0, 0.0, want_final=True)
    B, H, d = w.B, w.H, w.dk
    Hg, Gg = torch.empty(B, H, d, d, device="cuda"), torch.empty(B, H, d, d, device="cuda")
    o, it = gpu_forward(inp, w.dtype, w.cg_iters, 0.0, 64, H_final=Hg, G_final=Gg)
    forward_check(inp, o, it, w.dtype, w.cg_iters, 0.0, "full")
    for a, b in ((Hg, Hf), (Gg, Gf)):
        a = a.cpu().numpy().astype(np.float64)
        assert np.abs(a - b).max() <= 1e-5 * np.abs(b).max()
    # split the sequence: tokens [0, 70) then [70, 160) from the exported state
    t1 = 70
    first = {k: (v[:, :, :t1] if k != "lam" else v) for k, v in inp.items()}
    second = {k: (v[:, :, t1:] if k != "lam" else v) for k, v in inp.items()}
    H1, G1 = torch.empty_like(Hg), torch.empty_like(Gg)
    o1, _ = gpu_forward(first, w.dtype, w.cg_iters, 0.0, 32, H_final=H1, G_final=G1)
    o2, _ = gpu_forward(second, w.dtype, w.cg_iters, 0.0, 64, H0=H1, G0=G1)
    forward_check(inp, np.concatenate([o1, o2], axis=2), it, w.dtype, w.cg_iters, 0.0, "split")


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("f32", 16), ("bf16", 128)])
def test_unaligned_inputs(dtype, d):
    """q, k, v starting 4 (fp32) or 2 (bf16) bytes past a 16-byte boundary: fp32 d = 16 stays
    on the CUDA-core path and takes its element-wise loads (bit for bit the aligned result);
    fp32 d = 64 and bf16 d = 128 leave the tensor-core paths for the CUDA-core ones (checked
    against the oracle)."""
    import torch

    from mesa_layer_gb300 import binding
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    w = synth.workload("fwd_fp32_d64" if dtype == "f32" else "fwd_bf16_d128", B=1, H=2, T=100, dk=d, dv=d,
                       cg_tol=0.0, cg_iters=8)
    inp = synth.forward_inputs(w, seed=3)

    def shifted(x):
        flat = torch.from_numpy(np.ascontiguousarray(x)).to(td).reshape(-1)
        buf = torch.empty(flat.numel() + 1, dtype=td, device="cuda")
        view = buf[1:].view(x.shape)
        view.copy_(flat.view(x.shape))
        assert view.data_ptr() % 16 != 0
        return view

    al = {k: torch.from_numpy(inp[k]).cuda().to(td).contiguous() for k in ("q", "k", "v")}
    un = {k: shifted(inp[k]) for k in ("q", "k", "v")}
    g = torch.from_numpy(inp["gamma"]).cuda()
    lam = torch.from_numpy(inp["lam"]).cuda()
    o_al, i_al = binding.mesa_forward_chunked(al["q"], al["k"], al["v"], g, lam, 8, 0.0, w.chunk)
    out_un = torch.empty((1, 2, 100, d), dtype=td, device="cuda")
    o_un, i_un = binding.mesa_forward_chunked(un["q"], un["k"], un["v"], g, lam, 8, 0.0, w.chunk, out=out_un)
    torch.cuda.synchronize()
    assert torch.equal(i_al, i_un)
    if dtype == "f32" and d == 16:
        assert torch.equal(o_al, o_un)
    elif dtype == "f32":
        r = forward_check(inp, o_un.float().cpu().numpy(), i_un.cpu().numpy(), "f32", 8, 0.0, "unaligned f32")
        print(f"unaligned f32 d={d} (CUDA-core path): {r}")
    else:
        # the CUDA-core fp32 path with 8 unconverged iterations: one token's readout cancels
        # (strict 5.1e-2, 1.3e-4 on the readout's magnitude), as fp32 arithmetic predicts
        r = forward_check(inp, o_un.float().cpu().numpy(), i_un.cpu().numpy(), "bf16", 8, 0.0, "unaligned",
                          metric="product")
        print(f"unaligned bf16 (CUDA-core path): {r}")
