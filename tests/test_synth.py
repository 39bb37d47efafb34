"""Host-side checks of the seeded input generators (no GPU)."""
import numpy as np

from mesa_layer_gb300 import synth


def test_bf16_rounding_ties_to_even_and_exactness():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 2**-7 + 2**-8, 3.14159, -2.5e-3, 0.0], dtype=np.float32)
    r = synth.round_bf16(x)
    assert r[0] == 1.0 and r[1] == 1.0                      # tie -> even
    assert r[2] == np.float32(1.0 + 2**-6)                  # tie -> even (upwards)
    bits = r.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)
    assert np.all(np.abs(r - x) <= np.abs(x) * 2**-8 + 1e-30)
    assert np.array_equal(synth.round_bf16(r), r)


def test_forward_inputs_shapes_determinism_and_distributions():
    w = synth.workload("fwd_fp32_d64", B=1, H=2, T=128)
    a = synth.forward_inputs(w, seed=0)
    b = synth.forward_inputs(w, seed=0)
    c = synth.forward_inputs(w, seed=1)
    for key in a:
        assert np.array_equal(a[key], b[key])
        assert a[key].dtype == np.float32
    assert not np.array_equal(a["q"], c["q"])
    assert a["q"].shape == (1, 2, 128, 64) and a["lam"].shape == (2, 64)
    np.testing.assert_allclose(np.linalg.norm(a["k"], axis=-1), 1.0, rtol=1e-5)
    assert np.all((a["gamma"] > 0) & (a["gamma"] < 1))
    assert np.all((a["lam"] >= 0.1) & (a["lam"] <= 1.0))


def test_bf16_workload_inputs_are_bf16_values():
    w = synth.workload("fwd_bf16_d128", B=1, H=1, T=64)
    a = synth.forward_inputs(w)
    for key in ("q", "k", "v"):
        assert np.all(a[key].view(np.uint32) & 0xFFFF == 0)


def test_decode_inputs_per_step_streams():
    w = synth.workload("decode_bf16_d128", B=4, H=2)
    s0 = synth.decode_inputs(w, 0)
    s1 = synth.decode_inputs(w, 1)
    p = synth.decode_inputs(w, -w.prefix)
    assert s0["q"].shape == (4, 2, 128) and s0["gamma"].shape == (4, 2)
    assert not np.array_equal(s0["k"], s1["k"]) and not np.array_equal(s0["k"], p["k"])
    assert np.array_equal(synth.decode_inputs(w, 1)["v"], s1["v"])


def test_backward_inputs_add_an_independent_gradient_stream():
    w = synth.workload("bwd_bf16_d128", B=1, H=2, T=96)
    a = synth.backward_inputs(w, seed=0)
    f = synth.forward_inputs(w, seed=0)
    for key in ("q", "k", "v", "gamma", "lam"):
        assert np.array_equal(a[key], f[key])          # the forward's inputs, unchanged
    assert a["dout"].shape == (1, 2, 96, 128) and a["dout"].dtype == np.float32
    assert np.all(a["dout"].view(np.uint32) & 0xFFFF == 0)   # bf16 values
    assert np.array_equal(synth.backward_inputs(w, seed=0)["dout"], a["dout"])
    assert not np.array_equal(synth.backward_inputs(w, seed=1)["dout"], a["dout"])
    assert not np.allclose(a["dout"], a["v"])          # its own stream, not v's
    assert abs(float(a["dout"].std()) - 1.0) < 0.05
