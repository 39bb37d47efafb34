"""Pins of the oracle's backward pass (gradients through the Mesa layer).

The pages claim training ("Paralelizacao" bullet: O(T) training; "Contribuicoes", item 1) but
give no gradient.  Reading: implicit differentiation through each token's solve: with
g_t = dL/do_t, b_t = G_t^T g_t and y_t = CG(H_t + Lambda, b_t) (the forward's CG rule), dq_t =
y_t, the state gradients -y_t x_t^T and g_t x_t^T, and the state recurrence differentiated
backwards in time.

Checked against things other than the oracle itself: central finite differences of the
forward oracle run to convergence (per element on a tiny case, along random directions on a
case longer than the backward sweep's 64-token stretches), autograd of an independent dense
formulation in torch (states from explicit decay products, not the recurrence; an exact
solve), the one-token Sherman-Morrison closed form, and the dynamic stopping rule of the
second solve against the true residual.  Planted mistakes must each fail the battery."""
import os

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "mesa_oracle.c")


def _case(rng, B, H, T, d, glo=0.8):
    q = rng.standard_normal((B, H, T, d))
    k = rng.standard_normal((B, H, T, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, d))
    g = rng.uniform(glo, 1.0, (B, H, T))
    lam = rng.uniform(0.3, 1.0, (H, d))
    do = rng.standard_normal((B, H, T, d))
    return q, k, v, g, lam, do


def _loss(lib, q, k, v, g, lam, do, iters):
    o, _ = oracle.forward(q, k, v, g, lam, iters, lib=lib, nthreads=1)
    return float((o * do).sum())


NAMES = (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dgamma"), ("lam", "dlam"))


def _fd_elements(lib, case, iters, h=1e-6):
    q, k, v, g, lam, do = case
    args = {"q": q, "k": k, "v": v, "g": g, "lam": lam}
    out = {}
    for name, _ in NAMES:
        arr = args[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += h
            a2[idx] -= h
            l1 = _loss(lib, **{**args, name: a1}, do=do, iters=iters)
            l2 = _loss(lib, **{**args, name: a2}, do=do, iters=iters)
            fd[idx] = (l1 - l2) / (2 * h)
        out[name] = fd
    return out


def _battery(lib) -> list:
    """Names of the backward pins that fail for this compiled copy of the oracle."""
    failed = []
    rng = np.random.default_rng(21)
    # (1) per-element central differences; CG with d iterations is the exact solve
    d = 3
    case = _case(rng, 1, 2, 6, d)
    r = oracle.backward(*case, cg_iters=d, lib=lib, nthreads=1)
    fd = _fd_elements(lib, case, d)
    for name, key in NAMES:
        scale = max(np.abs(fd[name]).max(), 1e-12)
        if np.abs(fd[name] - r[key]).max() > 1e-6 * scale:
            failed.append(f"fd_{name}")
    # (2) directional differences on 150 tokens (three backward stretches)
    case = _case(rng, 1, 1, 150, d, glo=0.9)
    q, k, v, g, lam, do = case
    r = oracle.backward(*case, cg_iters=d, lib=lib, nthreads=1)
    args = {"q": q, "k": k, "v": v, "g": g, "lam": lam}
    h = 1e-6
    for name, key in NAMES:
        dirn = rng.standard_normal(args[name].shape)
        l1 = _loss(lib, **{**args, name: args[name] + h * dirn}, do=do, iters=d)
        l2 = _loss(lib, **{**args, name: args[name] - h * dirn}, do=do, iters=d)
        fdd = (l1 - l2) / (2 * h)
        an = float((r[key] * dirn).sum())
        if abs(fdd - an) > 1e-6 * max(abs(fdd), 1.0):
            failed.append(f"dir_{name}")
    # (3) one token, A = k k^T + Lambda: Sherman-Morrison,
    # A^-1 z = L^-1 z - L^-1 k (k . L^-1 z) / (1 + k . L^-1 k); the gate has no earlier state
    rng1 = np.random.default_rng(5)
    d1 = 5
    q, k, v, g, lam, do = _case(rng1, 1, 1, 1, d1)
    r = oracle.backward(q, k, v, g, lam, do, cg_iters=d1, lib=lib, nthreads=1)
    kk, qq, vv, gg, ll = k[0, 0, 0], q[0, 0, 0], v[0, 0, 0], do[0, 0, 0], lam[0]
    den = 1.0 + kk @ (kk / ll)
    dq_cf = (kk / ll) * (vv @ gg) / den              # A^-1 k (v.g), A = k k^T + Lambda
    x_cf = qq / ll - (kk / ll) * (kk @ (qq / ll)) / den
    dv_cf = gg * (kk @ (qq / ll)) / den              # g (k . A^-1 q)
    if not (np.allclose(r["dq"][0, 0, 0], dq_cf, rtol=1e-10, atol=1e-13)
            and np.allclose(r["dv"][0, 0, 0], dv_cf, rtol=1e-10, atol=1e-13)
            and np.allclose(r["dlam"][0], -dq_cf * x_cf, rtol=1e-10, atol=1e-13)
            and r["dgamma"][0, 0, 0] == 0.0):
        failed.append("sherman_morrison")
    # (4) dynamic mode: the second solve stops at the first count whose true residual
    # ||b - A y|| meets tol ||b||, b = G_t^T g_t from the oracle's state trace
    rng2 = np.random.default_rng(8)
    d2 = 8
    q, k, v, g, lam, do = _case(rng2, 1, 1, 12, d2)
    tol = 1e-3
    r = oracle.backward(q, k, v, g, lam, do, cg_iters=40, cg_tol=tol, lib=lib, nthreads=1)
    Ha, Ga = oracle.state_trace(k[0, 0], v[0, 0], g[0, 0], lib=lib)
    for t in range(12):
        A = Ha[t] + np.diag(lam[0])
        b = Ga[t].T @ do[0, 0, t]
        n = int(r["iters_bwd"][0, 0, t])
        y = r["dq"][0, 0, t]
        lim = tol * np.linalg.norm(b)
        ym, _ = oracle.cg(Ha[t], lam[0], b, max(n - 1, 0), lib=lib)
        if np.linalg.norm(b - A @ y) > lim * (1 + 1e-3) or (n > 0 and np.linalg.norm(b - A @ ym) <= lim * (1 - 1e-3)):
            failed.append("dynamic_second_solve")
            break
    return failed


def test_battery_passes_on_the_real_oracle():
    assert _battery(oracle.load()) == []


def test_dense_autograd_formulation():
    """torch autograd of an independent dense formulation: H_t and G_t as explicit sums with
    decay products prod_{s=t'+1..t} gamma_s, o_t = G_t (H_t + Lambda)^-1 q_t by an exact
    solve; the oracle's CG runs d iterations (exact)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(33)
    B, H, T, d = 2, 2, 9, 4
    q, k, v, g, lam, do = _case(rng, B, H, T, d)
    r = oracle.backward(q, k, v, g, lam, do, cg_iters=d)
    tq, tk, tv, tg, tl = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v, g, lam))
    loss = torch.zeros((), dtype=torch.float64)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                Hm = torch.zeros((d, d), dtype=torch.float64)
                Gm = torch.zeros((d, d), dtype=torch.float64)
                for s in range(t + 1):
                    z = torch.prod(tg[b, h, s + 1:t + 1]) if s < t else torch.ones((), dtype=torch.float64)
                    Hm = Hm + z * torch.outer(tk[b, h, s], tk[b, h, s])
                    Gm = Gm + z * torch.outer(tv[b, h, s], tk[b, h, s])
                x = torch.linalg.solve(Hm + torch.diag(tl[h]), tq[b, h, t])
                loss = loss + torch.dot(Gm @ x, torch.tensor(do[b, h, t]))
    loss.backward()
    for t_, key in ((tq, "dq"), (tk, "dk"), (tv, "dv"), (tg, "dgamma"), (tl, "dlam")):
        ref = t_.grad.numpy()
        assert np.allclose(r[key], ref, rtol=1e-9, atol=1e-11 * np.abs(ref).max()), key


def test_fixed_mode_counts_and_zero_cotangent():
    rng = np.random.default_rng(2)
    q, k, v, g, lam, do = _case(rng, 2, 3, 20, 8)
    r = oracle.backward(q, k, v, g, lam, do, cg_iters=5)
    assert np.all(r["iters_fwd"] == 5) and np.all(r["iters_bwd"] == 5)
    z = oracle.backward(q, k, v, g, lam, np.zeros_like(do), cg_iters=5, cg_tol=1e-4)
    for key in ("dq", "dk", "dv", "dgamma", "dlam"):
        assert np.all(z[key] == 0.0), key
    assert np.all(z["iters_bwd"] == 0)  # b = 0 stops before the first iteration


MUTANTS = {
    "dk_without_transpose": ("(dH[(size_t)a * dk + c] + dH[(size_t)c * dk + a]) * kt[c]",
                             "(2.0 * dH[(size_t)a * dk + c]) * kt[c]"),
    "state_gradient_sign": ("for (int c = 0; c < dk; c++) dH[(size_t)a * dk + c] -= y[a] * x[c];",
                            "for (int c = 0; c < dk; c++) dH[(size_t)a * dk + c] += y[a] * x[c];"),
    "gate_gradient_drops_G": ("dgamma[tok] = dot((int)hh, dH, Hp) + dot((int)gg, dG, Gp);",
                              "dgamma[tok] = dot((int)hh, dH, Hp);"),
    "rhs_not_transposed": ("for (int a = 0; a < dv; a++) s += G[(size_t)a * dk + c] * g[a];",
                           "for (int a = 0; a < dv; a++) s += G[(size_t)c * dk + a] * g[a];"),
    "lambda_gradient_sign": ("dlam_u[(size_t)u * dk + c] -= y[c] * x[c];", "dlam_u[(size_t)u * dk + c] += y[c] * x[c];"),
    "stretch_state_not_restored": ("      memcpy(H, keepH + (size_t)(s0 / ORACLE_BWD_KEEP) * hh, sizeof(double) * hh);\n", ""),
    "adjoint_not_decayed": ("        for (size_t e = 0; e < hh; e++) dH[e] *= gamma[tok];\n", ""),
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
