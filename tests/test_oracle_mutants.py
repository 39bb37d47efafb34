"""Planted mistakes: each mutant of the oracle source (a plausible slip -- a dropped term, a
wrong sign, a wrong operand, an off-by-one in the forget factors) is compiled on the CPU
and must fail at least one pin.  This shows the pins can tell a wrong oracle from a
right one.  Pins are the same mathematics as test_oracle_pins.py, run on a small battery."""
import json
import os

import numpy as np
import pytest
import scipy.linalg

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "mesa_oracle.c")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_examples.json")

MUTANTS = {
    "no_decay_on_H": ("H[(size_t)a * dk + b] = gamma * H[(size_t)a * dk + b] + k[a] * k[b];",
                      "H[(size_t)a * dk + b] = H[(size_t)a * dk + b] + k[a] * k[b];"),
    "current_token_decayed": ("G[(size_t)a * dk + b] = gamma * G[(size_t)a * dk + b] + v[a] * k[b];",
                              "G[(size_t)a * dk + b] = gamma * (G[(size_t)a * dk + b] + v[a] * k[b]);"),
    "x_update_sign": ("x[i] += alpha * p[i];", "x[i] -= alpha * p[i];"),
    "r_update_sign": ("r[i] -= alpha * w[i];", "r[i] += alpha * w[i];"),
    "lambda_dropped": ("double s = lam[a] * p[a];", "double s = 0.0 * lam[a];"),
    "readout_uses_H": ("o[a] = dot(dk, G + (size_t)a * dk, x);", "o[a] = dot(dk, H + (size_t)a * dk, x);"),
    "beta_inverted": ("rho_next / rho : 0.0;", "rho / rho_next : 0.0;"),
    "stop_rule_too_strict": ("sqrt(rho) <= tol * qnorm", "sqrt(rho) <= 0.1 * tol * qnorm"),
}


def _explicit(k, v, gamma, t):
    H = np.zeros((k.shape[1], k.shape[1]))
    G = np.zeros((v.shape[1], k.shape[1]))
    for tp in range(t + 1):
        z = np.prod(gamma[tp + 1: t + 1])
        H += z * np.outer(k[tp], k[tp])
        G += z * np.outer(v[tp], k[tp])
    return H, G


def _battery(lib) -> list:
    """Returns the names of the pins that fail for this compiled copy of the oracle."""
    failed = []
    f1 = lambda q, k, v, g, lam, n, tol=0.0: [x[0, 0] for x in oracle.forward(
        q[None, None], k[None, None], v[None, None], g[None, None], lam[None], n, tol, lib=lib)]
    for case in json.load(open(GOLDEN))["cases"]:
        a = lambda key: np.array(case[key], dtype=np.float64)
        out, _ = f1(a("q"), a("k"), a("v"), a("gamma"), a("lam"), case["cg_iters"])
        if not np.allclose(out, a("out"), rtol=1e-12, atol=1e-13):
            failed.append("golden:" + case["name"])
    rng = np.random.default_rng(0)
    T, dk, dv = 8, 5, 3
    q, k, v = rng.standard_normal((T, dk)), rng.standard_normal((T, dk)), rng.standard_normal((T, dv))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    g = rng.uniform(0.6, 1.0, T)
    lam = rng.uniform(0.5, 1.5, dk)
    out, _ = f1(q, k, v, g, lam, dk)
    for t in range(T):
        H, G = _explicit(k, v, g, t)
        ref = G @ scipy.linalg.cho_solve(scipy.linalg.cho_factor(H + np.diag(lam)), q[t])
        if np.linalg.norm(out[t] - ref) > 1e-8 * np.linalg.norm(ref):
            failed.append("cholesky")
            break
    out, it = f1(q, k, v, g, lam, 50, 1e-3)
    for t in range(T):
        H, _ = _explicit(k, v, g, t)
        A = H + np.diag(lam)
        n = int(it[t])
        xn, _ = oracle.cg(H, lam, q[t], n)
        xm, _ = oracle.cg(H, lam, q[t], max(n - 1, 0))
        tol = 1e-3 * np.linalg.norm(q[t])
        if np.linalg.norm(q[t] - A @ xn) > tol * (1 + 1e-6) or (
                n > 0 and np.linalg.norm(q[t] - A @ xm) <= tol * (1 - 1e-6)):
            failed.append("dynamic_stop")
            break
    return failed


def test_battery_passes_on_the_real_oracle():
    assert _battery(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.load(oracle.compile_oracle(str(mpath), str(tmp_path / "libmutant.so")))
    assert _battery(lib), f"planted mistake {name} went unnoticed"
