"""GPU parity of the query/key preprocessing (mesa_qk_preprocess and mesa_qk_preprocess_step
through the C ABI) against the fp64 oracle: every channel count and window, ragged lengths,
zero inputs, decode steps against the sequence form, the prefill-to-decode hand-off, and the
full-size workload on sampled units.

The outputs are unit vectors, so the unit metric (largest absolute error over largest
absolute reference value of a (batch, head) sequence) is bounded by the output rounding:
~1e-7 in fp32, 2^-9 in bf16."""
import numpy as np
import pytest

import oracle
from mesa_layer_gb300 import synth
from helpers import TOL, token_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mesa_layer_gb300 import binding, build
    build.build()
    binding.load()


def _dev(inp, dtype):
    import torch
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    return {k: torch.from_numpy(np.ascontiguousarray(v)).cuda().to(td if k.endswith("_raw") else torch.float32)
            .contiguous() for k, v in inp.items()}


def _check(o_gpu, o_ref, dtype, label):
    """Strict per-token error (each output token is a unit vector or zero)."""
    err = token_err(o_gpu.reshape(-1, *o_gpu.shape[-2:]), o_ref.reshape(-1, *o_ref.shape[-2:])).max()
    print(f"{label}: strict per-token max {err:.3e}")
    assert err <= TOL[dtype], f"{label}: {err:.3e}"
    return err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("W", [1, 2, 4, 8])
def test_sequence_against_oracle(dtype, d, W):
    from mesa_layer_gb300 import binding
    w = synth.workload("qkpre_bf16_d128", dtype=dtype, B=2, H=3, T=301, dk=d, dv=d)
    inp = synth.preprocess_inputs(w, taps=W, seed=d + W)
    t = _dev(inp, dtype)
    qo, ko = binding.mesa_qk_preprocess(t["q_raw"], t["k_raw"], t["wq"], t["wk"])
    for name, o, raw, wt in (("q", qo, "q_raw", "wq"), ("k", ko, "k_raw", "wk")):
        ref = oracle.qk_preprocess(inp[raw], inp[wt])
        _check(o.float().cpu().numpy(), ref, dtype, f"pre {name} d={d} W={W} {dtype}")


def test_zero_tokens_stay_zero():
    import torch

    from mesa_layer_gb300 import binding
    w = synth.workload("qkpre_bf16_d128", dtype="f32", B=1, H=2, T=40, dk=64, dv=64)
    inp = synth.preprocess_inputs(w, taps=3, seed=1)
    inp["q_raw"][:, :, 10:20] = 0.0          # a zero stretch longer than the window
    t = _dev(inp, "f32")
    qo, _ = binding.mesa_qk_preprocess(t["q_raw"], t["k_raw"], t["wq"], t["wk"])
    q = qo.cpu().numpy()
    assert np.all(q[:, :, 12:20] == 0.0)     # the window saw only zeros
    assert np.allclose(np.linalg.norm(q[:, :, 20:], axis=-1), 1.0, atol=1e-6)
    ref = oracle.qk_preprocess(inp["q_raw"], inp["wq"])
    _check(q, ref, "f32", "pre zero stretch")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_steps_match_the_sequence_and_the_prefill_hands_over(dtype):
    """A prefill of T0 tokens, then decode steps from a window holding the prefill's last
    W-1 raw inputs, give the preprocessing of the whole sequence."""
    import torch

    from mesa_layer_gb300 import binding
    W, T0, T1 = 4, 13, 9
    w = synth.workload("qkpre_bf16_d128", dtype=dtype, B=3, H=2, T=T0 + T1, dk=128, dv=128)
    inp = synth.preprocess_inputs(w, taps=W, seed=7)
    t = _dev(inp, dtype)
    ref_q = oracle.qk_preprocess(inp["q_raw"], inp["wq"])
    ref_k = oracle.qk_preprocess(inp["k_raw"], inp["wk"])
    qp, kp = binding.mesa_qk_preprocess(t["q_raw"][:, :, :T0].contiguous(), t["k_raw"][:, :, :T0].contiguous(),
                                        t["wq"], t["wk"])
    # window after the prefill: [N, H, 2, W-1, d], entry s = input s+1 tokens back
    state = torch.zeros((w.B, w.H, 2, W - 1, w.dk), device="cuda")
    for s in range(W - 1):
        state[:, :, 0, s] = t["q_raw"][:, :, T0 - 1 - s].float()
        state[:, :, 1, s] = t["k_raw"][:, :, T0 - 1 - s].float()
    qs, ks = [], []
    for step in range(T1):
        qo, ko = binding.mesa_qk_preprocess_step(t["q_raw"][:, :, T0 + step].contiguous(),
                                                 t["k_raw"][:, :, T0 + step].contiguous(), t["wq"], t["wk"], state)
        qs.append(qo.float().cpu().numpy())
        ks.append(ko.float().cpu().numpy())
    q = np.concatenate([qp.float().cpu().numpy(), np.stack(qs, axis=2)], axis=2)
    k = np.concatenate([kp.float().cpu().numpy(), np.stack(ks, axis=2)], axis=2)
    _check(q, ref_q, dtype, f"pre prefill+steps q {dtype}")
    _check(k, ref_k, dtype, f"pre prefill+steps k {dtype}")
    # and from an empty window the steps reproduce the GPU's own sequence form bit for bit
    state.zero_()
    qseq, _ = binding.mesa_qk_preprocess(t["q_raw"], t["k_raw"], t["wq"], t["wk"])
    for step in range(5):
        qo, _ = binding.mesa_qk_preprocess_step(t["q_raw"][:, :, step].contiguous(),
                                                t["k_raw"][:, :, step].contiguous(), t["wq"], t["wk"], state)
        assert torch.equal(qo, qseq[:, :, step])


def test_full_workload_sampled_units():
    """The benchmark's preprocessing workload (B=8 H=16 T=4096 d=128 W=4, bf16); the oracle
    follows three (batch, head) units."""
    from mesa_layer_gb300 import binding
    w = synth.workload("qkpre_bf16_d128")
    inp = synth.preprocess_inputs(w, seed=0)
    t = _dev(inp, w.dtype)
    qo, ko = binding.mesa_qk_preprocess(t["q_raw"], t["k_raw"], t["wq"], t["wk"])
    for b, h in ((0, 0), (3, 7), (7, 15)):
        for name, o, raw, wt in (("q", qo, "q_raw", "wq"), ("k", ko, "k_raw", "wk")):
            x = inp[raw][b:b + 1, h:h + 1]
            ref = oracle.qk_preprocess(x, inp[wt][h:h + 1])
            _check(o[b:b + 1, h:h + 1].float().cpu().numpy(), ref, w.dtype, f"pre full {name} b={b} h={h}")

