"""GPU parity of the recurrent decode step (mesa_decode_step through the C ABI) against
the fp64 oracle, including the full-size decode workload on sampled units."""
import numpy as np
import pytest

import oracle
from mesa_layer_gb300 import synth
from helpers import check_against_oracle, oracle_decode_units

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


def _run(w, steps, prefix, units=None, iters=None, tol=None, metric=None):
    """Decode `prefix` state-only steps (cg_iters = 0) and then `steps` full steps on the GPU
    and, for `units` (list of (n, h); default all), in the oracle; every step's output of
    every sampled unit is checked per token (dynamic mode: against the oracle replaying the
    GPU's count where the two stopping decisions differ).  Returns (Result, count agreement)."""
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
    units = units or [(n, h) for n in range(N) for h in range(H)]
    nidx = np.array([u[0] for u in units])
    hidx = np.array([u[1] for u in units])
    U = len(units)
    Ho = np.zeros((U, 1, d, d))
    Go = np.zeros((U, 1, d, d))
    lam_u = lam[hidx]  # each sampled unit keeps its head's lambda (as a 1-head oracle unit)
    acc = {k: [] for k in ("og", "ig", "ro", "rit", "rr", "rs")}
    for s in range(-prefix, steps):
        inp = synth.decode_inputs(w, s)
        dev = {k: torch.from_numpy(inp[k]).cuda().to(td if k != "gamma" else torch.float32)
               for k in ("q", "k", "v", "gamma")}
        n_it = 0 if s < 0 else iters
        o, it = binding.mesa_decode_step(Hs, Gs, dev["q"], dev["k"], dev["v"], dev["gamma"], lam_t, n_it, tol)
        if s < 0:
            oracle_decode_units(Ho, Go, inp, nidx, hidx, lam_u, 0, tol)
            continue
        torch.cuda.synchronize()
        ig = it.cpu().numpy()[nidx, hidx]
        ro, rit, rr, rs = oracle_decode_units(Ho, Go, inp, nidx, hidx, lam_u, n_it, tol, gpu_counts=ig)
        for k, v in (("og", o.float().cpu().numpy()[nidx, hidx]), ("ig", ig), ("ro", ro), ("rit", rit),
                     ("rr", rr), ("rs", rs)):
            acc[k].append(v)
    Hg = Hs.cpu().numpy()[nidx, hidx]
    Gg = Gs.cpu().numpy()[nidx, hidx]
    assert np.abs(Hg - Ho[:, 0]).max() <= 1e-5 * np.abs(Ho).max()
    assert np.abs(Gg - Go[:, 0]).max() <= 1e-5 * np.abs(Go).max()
    # per unit over its steps: arrays [U, steps, d] and [U, steps]
    a = {k: np.stack(v, axis=1) for k, v in acc.items()}
    # scale of the oracle's own run: only used when the counts all agree (then rr == ro)
    r = check_against_oracle(a["og"], a["ig"], a["ro"], a["rit"], a["rs"], w.dtype, tol, "decode",
                             replay=lambda counts: (a["rr"], a["rs"]), metric=metric)
    return r, a["ig"] == a["rit"]


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_small(d, dtype):
    w = synth.workload("decode_bf16_d128", B=3, H=2, dk=d, dv=d, dtype=dtype, prefix=0)
    r, agree = _run(w, steps=24, prefix=0, iters=d + 4, tol=0.0)
    print(f"decode d={d} {dtype}: {r}")


@pytest.mark.parametrize("d", [64, 128])
def test_decode_scale_is_exact(d):
    """The step is homogeneous: q times 2^k scales x and o; v and G_state times 2^k scale o and
    the new G_state; H_state is untouched by either.  In fp32 arithmetic with power-of-two
    factors every result is exactly 2^k times the unscaled one (k = -40, 40), with the same
    counts, in fixed and dynamic mode (the stopping rule compares norms that scale alike)."""
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload("decode_bf16_d128", B=3, H=2, dk=d, dv=d, prefix=0)
    N, H = w.B, w.H
    lam_t = torch.from_numpy(synth.lambdas(w)).cuda()
    rng = np.random.default_rng(21)
    M = rng.standard_normal((N, H, d, d)).astype(np.float32) * 0.1
    H0 = torch.from_numpy((M @ np.swapaxes(M, -1, -2)).astype(np.float32)).cuda()
    G0 = torch.from_numpy((rng.standard_normal((N, H, d, d)) * 0.1).astype(np.float32)).cuda()
    inp = synth.decode_inputs(w, 0)
    dev = {k: torch.from_numpy(inp[k]).cuda().to(torch.bfloat16 if k != "gamma" else torch.float32)
           for k in ("q", "k", "v", "gamma")}
    for iters, tol in ((d // 2, 0.0), (30, 1e-3)):
        Hb, Gb = H0.clone(), G0.clone()
        o, it = binding.mesa_decode_step(Hb, Gb, dev["q"], dev["k"], dev["v"], dev["gamma"], lam_t, iters, tol)
        for k in (-40, 40):
            f = 2.0 ** k
            Hq, Gq = H0.clone(), G0.clone()
            oq, itq = binding.mesa_decode_step(Hq, Gq, dev["q"] * f, dev["k"], dev["v"], dev["gamma"], lam_t, iters, tol)
            Hv, Gv = H0.clone(), (G0 * f).contiguous()
            ov, itv = binding.mesa_decode_step(Hv, Gv, dev["q"], dev["k"], dev["v"] * f, dev["gamma"], lam_t, iters, tol)
            torch.cuda.synchronize()
            for o2, it2 in ((oq, itq), (ov, itv)):
                assert torch.equal(it2, it), (iters, k)
                assert torch.equal(o2.float(), o.float() * f), (iters, k)
            assert torch.equal(Hq, Hb) and torch.equal(Gq, Gb) and torch.equal(Hv, Hb), (iters, k)
            assert torch.equal(Gv, Gb * f), (iters, k)


def test_decode_dynamic_with_prefix():
    # fp32 inputs and the 1e-4 tolerance of fp32 workloads: Lambda >= 0.5 keeps the systems
    # well enough conditioned for fp32 CG to track the fp64 iterates at that level
    w = synth.workload("decode_bf16_d128", B=4, H=2, dtype="f32", prefix=40, lam_lo=0.5, lam_hi=1.0)
    r, agree = _run(w, steps=16, prefix=40, tol=1e-4)
    print(f"decode dynamic: {r}")


def test_decode_full_size_sampled_units():
    w = synth.workload("decode_bf16_d128")
    units = [(0, 0), (17, 5), (128, 9), (255, 15)]
    r, agree = _run(w, steps=w.decode_steps, prefix=w.prefix, units=units)
    print(f"decode full: {r}")
