"""Pins of the oracle's warm-started CG (the pages' remark, "Significancia", that warm-start
strategies could cut the CG cost; reading: the decode step's CG starts from the previous
step's solution, r0 = q - (H + Lambda) x0, and the stopping rule stays relative to ||q||).

Checked against: the cold CG (x0 = 0), the dense Cholesky solve (finite termination from any
start), the one-step closed form, the exact solution as a start (no iteration needed), the
true residual at the stopping point, and the decode-step bookkeeping of the start vector.
Planted mistakes must each fail the battery."""
import os

import numpy as np
import pytest
import scipy.linalg

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "mesa_oracle.c")


def _spd(rng, n):
    K = rng.standard_normal((3 * n, n))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    g = rng.uniform(0.8, 1.0, 3 * n)
    H = np.zeros((n, n))
    for t in range(3 * n):
        H = g[t] * H + np.outer(K[t], K[t])
    return H, rng.uniform(0.2, 1.0, n)


def _battery(lib) -> list:
    failed = []
    rng = np.random.default_rng(11)
    n = 6
    H, lam = _spd(rng, n)
    A = H + np.diag(lam)
    q = rng.standard_normal(n)
    x0 = rng.standard_normal(n)
    xs = scipy.linalg.cho_solve(scipy.linalg.cho_factor(A), q)
    # a zero start is the cold CG, bit for bit
    xc, ic = oracle.cg(H, lam, q, 4, lib=lib)
    xz, iz = oracle.cg(H, lam, q, 4, x0=np.zeros(n), lib=lib)
    if not (np.array_equal(xc, xz) and ic == iz):
        failed.append("zero_start")
    # n iterations from any start reach the exact solve
    xn, _ = oracle.cg(H, lam, q, n, x0=x0, lib=lib)
    if np.linalg.norm(xn - xs) > 1e-9 * np.linalg.norm(xs):
        failed.append("finite_termination")
    # one iteration: x1 = x0 + alpha r0, alpha = r0.r0 / r0.A r0
    r0 = q - A @ x0
    x1_ref = x0 + (r0 @ r0) / (r0 @ A @ r0) * r0
    x1, _ = oracle.cg(H, lam, q, 1, x0=x0, lib=lib)
    if np.linalg.norm(x1 - x1_ref) > 1e-12 * np.linalg.norm(x1_ref):
        failed.append("one_step")
    # starting at the solution: no iteration in dynamic mode, the start is returned
    xw, iw = oracle.cg(H, lam, q, 20, tol=1e-6, x0=xs, lib=lib)
    if iw != 0 or not np.array_equal(xw, xs):
        failed.append("start_at_solution")
    # dynamic stop: the true residual meets tol ||q|| at the returned count, not one earlier
    tol = 1e-4
    xd, idn = oracle.cg(H, lam, q, 50, tol=tol, x0=x0, lib=lib)
    xm, _ = oracle.cg(H, lam, q, max(idn - 1, 0), x0=x0, lib=lib)
    lim = tol * np.linalg.norm(q)
    if np.linalg.norm(q - A @ xd) > lim * (1 + 1e-6) or (idn > 0 and np.linalg.norm(q - A @ xm) <= lim * (1 - 1e-6)):
        failed.append("dynamic_stop")
    # decode step: the start vector is read and replaced by the solution of this step
    N, heads, dk, dv = 1, 2, n, 3
    Hs = np.zeros((N, heads, dk, dk))
    Gs = np.zeros((N, heads, dv, dk))
    Hs[0, 0], Hs[0, 1] = H, H.T
    X = np.ascontiguousarray(rng.standard_normal((N, heads, dk)))
    X_in = X.copy()
    qq = rng.standard_normal((N, heads, dk))
    kk = rng.standard_normal((N, heads, dk))
    vv = rng.standard_normal((N, heads, dv))
    gg = np.array([[0.9, 0.95]])
    lam2 = np.stack([lam, lam[::-1]])
    Hc, Gc = Hs.copy(), Gs.copy()
    out, it = oracle.decode_step(Hc, Gc, qq, kk, vv, gg, lam2, 3, 0.0, X=X, lib=lib)
    for h in range(heads):
        Hn = gg[0, h] * Hs[0, h] + np.outer(kk[0, h], kk[0, h])
        xr, _ = oracle.cg(Hn, lam2[h], qq[0, h], 3, x0=X_in[0, h], lib=lib)
        Gn = gg[0, h] * Gs[0, h] + np.outer(vv[0, h], kk[0, h])
        if not (np.allclose(X[0, h], xr, rtol=1e-13, atol=1e-15) and np.allclose(out[0, h], Gn @ xr, rtol=1e-12, atol=1e-14)):
            failed.append("decode_start_vector")
            break
    return failed


def test_battery_passes_on_the_real_oracle():
    assert _battery(oracle.load()) == []


MUTANTS = {
    "start_ignored_in_residual": ("      r[i] = q[i] - w[i];\n", "      r[i] = q[i] + 0.0 * w[i];\n"),
    "iterate_not_from_start": ("      x[i] = x0[i];\n", "      x[i] = 0.0;\n"),
    "stop_relative_to_r0": ("const double qnorm = x0 ? sqrt(dot(n, q, q)) : sqrt(rho);", "const double qnorm = sqrt(rho);"),
    "start_not_replaced": ("    if (xu) memcpy(xu, x, sizeof(double) * dk);\n", ""),
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
