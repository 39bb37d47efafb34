"""GPU parity of the warm-started decode step (mesa_decode_step_warm through the C ABI): each
unit's CG starts from the previous step's solution, carried in a caller-owned start-vector
state.  Against the fp64 oracle's warm-started decode step (outputs, the carried start
vectors, iteration counts), and a zero start against the cold decode step bit for bit."""
import numpy as np
import pytest

import oracle
from mesa_layer_gb300 import synth
from helpers import TOL, check_against_oracle, oracle_decode_units, unit_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


def _dev(inp, td):
    import torch
    return {k: torch.from_numpy(inp[k]).cuda().to(td if k != "gamma" else torch.float32) for k in ("q", "k", "v", "gamma")}


def _run(w, steps, prefix, units=None, iters=None, tol=None):
    """`prefix` state-only steps, then `steps` warm-started steps on the GPU and, for the
    sampled units, in the oracle (each unit a one-head oracle unit with its head's lambda)."""
    import torch

    from mesa_layer_gb300 import binding
    iters = w.cg_iters if iters is None else iters
    tol = w.cg_tol if tol is None else tol
    N, H, d = w.B, w.H, w.dk
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    lam = synth.lambdas(w)
    lam_t = torch.from_numpy(lam).cuda()
    Hs = torch.zeros(N, H, d, d, device="cuda")
    Gs = torch.zeros(N, H, d, d, device="cuda")
    Xs = torch.zeros(N, H, d, device="cuda")
    units = units or [(n, h) for n in range(N) for h in range(H)]
    nidx = np.array([u[0] for u in units])
    hidx = np.array([u[1] for u in units])
    U = len(units)
    Ho, Go = np.zeros((U, 1, d, d)), np.zeros((U, 1, d, d))
    Xo = np.zeros((U, 1, d))
    lam_u = lam[hidx]
    acc = {k: [] for k in ("og", "ig", "ro", "rit", "rr", "rs")}
    xerr = 0.0
    for s in range(-prefix, steps):
        inp = synth.decode_inputs(w, s)
        dev = _dev(inp, td)
        if s < 0:  # state-only prefix (no CG; the start vectors stay zero)
            binding.mesa_decode_step(Hs, Gs, dev["q"], dev["k"], dev["v"], dev["gamma"], lam_t, 0, tol)
            oracle_decode_units(Ho, Go, inp, nidx, hidx, lam_u, 0, tol)
            continue
        o, it = binding.mesa_decode_step_warm(Hs, Gs, Xs, dev["q"], dev["k"], dev["v"], dev["gamma"], lam_t, iters, tol)
        torch.cuda.synchronize()
        ig = it.cpu().numpy()[nidx, hidx]
        # the oracle's start vectors follow the GPU's counts (replayed where they differ)
        ro, rit, rr, rs = oracle_decode_units(Ho, Go, inp, nidx, hidx, lam_u, iters, tol, gpu_counts=ig, Xo=Xo)
        for k, v in (("og", o.float().cpu().numpy()[nidx, hidx]), ("ig", ig), ("ro", ro), ("rit", rit),
                     ("rr", rr), ("rs", rs)):
            acc[k].append(v)
        xg = Xs.cpu().numpy()[nidx, hidx]
        xerr = max(xerr, float(unit_err(xg[:, None], Xo[:, 0][:, None]).max()))
    a = {k: np.stack(v, axis=1) for k, v in acc.items()}
    r = check_against_oracle(a["og"], a["ig"], a["ro"], a["rit"], a["rs"], w.dtype, tol, "decode warm",
                             replay=lambda counts: (a["rr"], a["rs"]))
    return r, xerr, a["ig"], a["rit"]


def test_zero_start_is_the_cold_step():
    """With X_state = 0 the warm entry point runs exactly the cold CG (same outputs and
    counts, bit for bit) and leaves the solution in X_state."""
    import torch

    from mesa_layer_gb300 import binding
    for d in (64, 128):
        w = synth.workload("decode_bf16_d128", B=5, H=3, dk=d, dv=d)
        lam_t = torch.from_numpy(synth.lambdas(w)).cuda()
        H1 = torch.zeros(w.B, w.H, d, d, device="cuda")
        G1 = torch.zeros_like(H1)
        for s in range(-20, 0):
            x = _dev(synth.decode_inputs(w, s), torch.bfloat16)
            binding.mesa_decode_step(H1, G1, x["q"], x["k"], x["v"], x["gamma"], lam_t, 0, 0.0)
        H2, G2 = H1.clone(), G1.clone()
        X = torch.zeros(w.B, w.H, d, device="cuda")
        x = _dev(synth.decode_inputs(w, 0), torch.bfloat16)
        o1, i1 = binding.mesa_decode_step(H1, G1, x["q"], x["k"], x["v"], x["gamma"], lam_t, w.cg_iters, w.cg_tol)
        o2, i2 = binding.mesa_decode_step_warm(H2, G2, X, x["q"], x["k"], x["v"], x["gamma"], lam_t, w.cg_iters, w.cg_tol)
        assert torch.equal(o1, o2) and torch.equal(i1, i2) and torch.equal(H1, H2) and torch.equal(G1, G2)
        assert X.abs().max().item() > 0


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_warm_fixed_iterations(d, dtype):
    w = synth.workload("decode_bf16_d128", B=3, H=2, dk=d, dv=d, dtype=dtype, prefix=8)
    r, xerr, ig, rit = _run(w, steps=16, prefix=8, iters=6, tol=0.0)
    print(f"decode warm d={d} {dtype}: {r}, start vectors {xerr:.3e}")
    assert np.array_equal(ig, rit)
    assert xerr <= TOL[dtype]


def test_warm_dynamic_full_size_sampled_units():
    """The decode workload's shape and stopping rule with warm starts: 256 x 16 units, a
    64-step prefix, 24 warm steps, four units followed by the oracle."""
    w = synth.workload("decode_bf16_d128")
    units = [(0, 0), (17, 5), (128, 9), (255, 15)]
    r, xerr, ig, rit = _run(w, steps=24, prefix=64, units=units)
    agree = (ig == rit).mean()
    # (the start vectors are reported only: after a token whose count differs by one the two
    # sides carry starts that differ by up to the stopping tolerance's reach)
    print(f"decode warm full: {r}, start vectors {xerr:.3e}, counts agree {agree:.4f}, "
          f"mean iters {ig.mean():.2f} (oracle {rit.mean():.2f})")
