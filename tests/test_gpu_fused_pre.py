"""GPU parity of the query/key preprocessing fused into the chunked forward
(mesa_forward_chunked_pre through the C ABI): bit for bit against the two calls it replaces
(mesa_qk_preprocess, then mesa_forward_chunked; each is checked against the oracle on its own
inputs in test_gpu_preprocess.py and test_gpu_forward.py / test_gpu_tc.py), and end to end
against the fp64 oracle (oracle.qk_preprocess, rounded to the activations' dtype as the
preprocessing pass writes them, then oracle.forward).  MesaNet technical summary,
"Arquitetura (MesaNet)", "Pre-processamento"; "A Camada Mesa".

End to end, the layer's inputs are computed values: the GPU's fp32 preprocessing and the
oracle's fp64 one round to the same bf16 value except at near-ties (there they are one bf16
unit apart), and to fp32 values a unit or two apart.  The un-converged CG amplifies such
input differences by ~10^3, and a cancelling readout further still, so the end-to-end check
is made on the readout's magnitude (bf16: asserted at 2e-2; fp32: reported, the difference of
the two inputs being ~1e-7 x 10^3) and the dynamic cases' count agreement is reported with a
lower floor."""
import numpy as np
import pytest

import oracle
from mesa_layer_gb300 import synth
from helpers import forward_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


def _inputs(dtype, B, H, T, d, W, seed):
    w = synth.workload("fwd_bf16_d128", dtype=dtype, B=B, H=H, T=T, dk=d, dv=d)
    inp = synth.forward_inputs(w, seed=seed)
    inp.update(synth.preprocess_inputs(w, taps=W, seed=seed))
    return inp


def _dev(inp, dtype):
    import torch
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda().to(td if k in ("q_raw", "k_raw", "v") else torch.float32)
            .contiguous() for k, v in inp.items() if k not in ("q", "k")}


def _fused_and_two_pass(inp, dtype, iters, tol, chunk):
    import torch

    from mesa_layer_gb300 import binding
    t = _dev(inp, dtype)
    o1, i1 = binding.mesa_forward_chunked_pre(t["q_raw"], t["k_raw"], t["wq"], t["wk"], t["v"], t["gamma"], t["lam"],
                                              iters, tol, chunk)
    qp, kp = binding.mesa_qk_preprocess(t["q_raw"], t["k_raw"], t["wq"], t["wk"])
    o2, i2 = binding.mesa_forward_chunked(qp, kp, t["v"], t["gamma"], t["lam"], iters, tol, chunk)
    torch.cuda.synchronize()
    return o1, i1, o2, i2


def _oracle_inputs(inp, dtype):
    """The oracle's preprocessed q and k, rounded to the activations' dtype."""
    rnd = synth.round_bf16 if dtype == "bf16" else (lambda x: np.asarray(x, dtype=np.float32))
    sub = {k: inp[k] for k in ("v", "gamma", "lam")}
    sub["q"] = rnd(oracle.qk_preprocess(inp["q_raw"], inp["wq"]).astype(np.float32))
    sub["k"] = rnd(oracle.qk_preprocess(inp["k_raw"], inp["wk"]).astype(np.float32))
    return sub


CASES = [
    # (dtype, B, H, T, d, W, iters, tol)
    ("bf16", 1, 2, 300, 128, 4, 12, 0.0),            # tensor cores, ragged last chunk, window 4
    ("bf16", 2, 1, 128, 128, 1, 8, 0.0),             # window 1 (normalisation alone), one chunk
    ("bf16", 1, 1, 5, 128, 8, 6, 0.0),               # fewer tokens than the window
    ("bf16", 1, 3, 1000, 128, 3, 30, 1e-3),          # dynamic stopping
    ("bf16", 1, 1, 40 * 128 - 17, 128, 8, 10, 0.0),  # 40 chunks in segments, window 8
    ("f32", 2, 2, 200, 64, 4, 12, 0.0),              # CUDA cores: the pass, then the layer
    ("bf16", 1, 2, 150, 64, 2, 10, 1e-3),            # bf16, d = 64: the pass, then the layer
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_fused_equals_the_two_calls_and_the_oracle(case):
    import torch
    dtype, B, H, T, d, W, iters, tol = case
    inp = _inputs(dtype, B, H, T, d, W, seed=41)
    o1, i1, o2, i2 = _fused_and_two_pass(inp, dtype, iters, tol, 64)
    assert torch.equal(i1, i2) and torch.equal(o1, o2), "fused and two-pass results differ"
    r = forward_check(_oracle_inputs(inp, dtype), o1.float().cpu().numpy(), i1.cpu().numpy(), dtype, iters, tol,
                      str(case), metric="product", tol=(None if dtype == "bf16" else np.inf), min_agree=0.8)
    print(f"{case}: {r}")


def test_fused_full_size_bf16_d128_window4():
    """The 1B-scale layer shape (B=8, 16 heads, T=4096, d=128, fixed 15 iterations) with a
    4-tap window: bit for bit against the two calls everywhere; two sampled units against
    the oracle."""
    import torch
    w = synth.workload("fwd_bf16_d128")
    inp = _inputs("bf16", w.B, w.H, w.T, w.dk, 4, seed=0)
    o1, i1, o2, i2 = _fused_and_two_pass(inp, "bf16", w.cg_iters, 0.0, w.chunk)
    assert torch.equal(i1, i2) and torch.equal(o1, o2), "fused and two-pass results differ"
    o = o1.float().cpu().numpy()
    it = i1.cpu().numpy()
    for b, h in [(0, 0), (5, 9)]:
        unit = {k: inp[k][b, h][None, None] for k in ("q_raw", "k_raw", "v", "gamma")}
        unit["wq"], unit["wk"], unit["lam"] = inp["wq"][h][None], inp["wk"][h][None], inp["lam"][h][None]
        r = forward_check(_oracle_inputs(unit, "bf16"), o[b, h][None, None], it[b, h][None, None], "bf16",
                          w.cg_iters, 0.0, f"fused full ({b}, {h})")
        print(f"fused full ({b}, {h}): {r}")
