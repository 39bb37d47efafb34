"""Pins of the oracle's query/key preprocessing (MesaNet technical summary, section
"Arquitetura (MesaNet)", "Pre-processamento": keys and queries are normalised and convolved
with a small window before the Mesa layer).  Readings: a causal depthwise convolution over time
(W taps per head and channel, tap s multiplying the input s tokens back), then each token
divided by its Euclidean norm.

Each pin checks the oracle against something other than itself: numpy's full convolution, the
impulse response of the convolution, closed-form special cases, invariances, and the
sequence/step equivalence.  Planted mistakes (reversed taps, a non-causal window, normalising
before convolving, a dropped current tap, a wrong head) must each fail the battery."""
import os

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "mesa_oracle.c")


def _np_reference(x, w):
    """Full numpy convolution per (unit, channel), cut to the first T outputs (causal), then
    numpy's vector norm."""
    B, H, T, d = x.shape
    y = np.zeros_like(x)
    for b in range(B):
        for h in range(H):
            for c in range(d):
                y[b, h, :, c] = np.convolve(x[b, h, :, c], w[h, c, :])[:T]
    n = np.linalg.norm(y, axis=-1, keepdims=True)
    return np.where(n > 0, y / np.where(n > 0, n, 1.0), 0.0)


def _battery(lib) -> list:
    """Names of the preprocessing pins that fail for this compiled copy of the oracle."""
    failed = []
    rng = np.random.default_rng(3)
    B, H, T, d, W = 2, 3, 11, 5, 4
    x = rng.standard_normal((B, H, T, d))
    w = rng.standard_normal((H, d, W))
    out = oracle.qk_preprocess(x, w, lib=lib)
    if not np.allclose(out, _np_reference(x, w), rtol=1e-12, atol=1e-13):
        failed.append("numpy_convolve")
    # impulse in one channel of one unit: the output is sign(w[c, s]) e_c at t0 + s
    xi = np.zeros((1, 1, 9, 3))
    t0, c = 2, 1
    xi[0, 0, t0, c] = 2.5
    wi = np.array([[[0.5, -1.0, 2.0]] * 3])  # [1, 3, 3]
    oi = oracle.qk_preprocess(xi, wi, lib=lib)[0, 0]
    want = np.zeros((9, 3))
    for s in range(3):
        want[t0 + s, c] = np.sign(wi[0, c, s])
    if not np.allclose(oi, want, atol=1e-15):
        failed.append("impulse")
    # W = 1, unit tap: plain L2 normalisation, zero rows stay zero
    x1 = rng.standard_normal((1, 2, 6, 4))
    x1[0, 1, 3] = 0.0
    o1 = oracle.qk_preprocess(x1, np.ones((2, 4, 1)), lib=lib)
    n1 = np.linalg.norm(x1, axis=-1, keepdims=True)
    if not np.allclose(o1, np.where(n1 > 0, x1 / np.where(n1 > 0, n1, 1), 0), rtol=1e-13, atol=1e-15):
        failed.append("l2_only")
    # invariances: positive scaling of the input changes nothing, a sign flip flips the output
    if not np.allclose(oracle.qk_preprocess(7.0 * x, w, lib=lib), out, rtol=1e-12, atol=1e-14) or \
            not np.allclose(oracle.qk_preprocess(-x, w, lib=lib), -out, rtol=1e-12, atol=1e-14):
        failed.append("scale")
    # causality: a change at token t leaves earlier outputs alone and changes token t
    xc = x.copy()
    xc[:, :, 6] += 1.0
    oc = oracle.qk_preprocess(xc, w, lib=lib)
    if not np.array_equal(oc[:, :, :6], out[:, :, :6]) or np.allclose(oc[:, :, 6], out[:, :, 6]):
        failed.append("causal")
    # decode steps from an empty window reproduce the sequence
    hist = np.zeros((B, H, W - 1, d))
    steps = np.stack([oracle.qk_preprocess_step(x[:, :, t], w, hist, lib=lib) for t in range(T)], axis=2)
    if not np.allclose(steps, out, rtol=1e-13, atol=1e-15):
        failed.append("step_equals_sequence")
    return failed


def test_battery_passes_on_the_real_oracle():
    assert _battery(oracle.load()) == []


def test_unit_norm_rows():
    rng = np.random.default_rng(5)
    out = oracle.qk_preprocess(rng.standard_normal((2, 2, 40, 16)), rng.standard_normal((2, 16, 4)))
    assert np.allclose(np.linalg.norm(out, axis=-1), 1.0, atol=1e-13)


MUTANTS = {
    "taps_reversed": ("acc += wu[(size_t)c * W + s] * x[((size_t)u * T + (t - s)) * d + c];",
                      "acc += wu[(size_t)c * W + (W - 1 - s)] * x[((size_t)u * T + (t - s)) * d + c];"),
    "not_causal": ("for (int s = 0; s < W && s <= t; s++)\n          acc += wu[(size_t)c * W + s] * x[((size_t)u * T + (t - s)) * d + c];",
                   "for (int s = 0; s < W && t + s < T; s++)\n          acc += wu[(size_t)c * W + s] * x[((size_t)u * T + (t + s)) * d + c];"),
    "current_tap_dropped": ("for (int s = 0; s < W && s <= t; s++)", "for (int s = 1; s < W && s <= t; s++)"),
    "wrong_head": ("const double *wu = w + (size_t)(u % heads) * d * W;\n    for (int t = 0;",
                   "const double *wu = w + (size_t)(u / heads % heads) * d * W;\n    for (int t = 0;"),
    "norm_squared": ("const double n = sqrt(s);", "const double n = s;"),
    "step_history_not_shifted": ("    if (W > 1) memcpy(hu, xu, sizeof(double) * d);", ""),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.load(oracle.compile_oracle(str(mpath), str(tmp_path / "libmutant.so")))
    assert _battery(lib), f"planted mistake {name} went unnoticed"
