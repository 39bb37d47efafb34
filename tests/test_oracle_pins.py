"""Pins for the fp64 oracle: each test checks it against something other than itself.

Sources: MesaNet technical summary (gist.science/pt/paper/2506.05233), section "A Camada
Mesa" -- the Mesa objective (displayed equation), the readout Delta_t = Phi_t q_t through
q*_t = (H_t + Lambda)^-1 q_t solved by CG, the state variables G_t/H_t ("Paralelizacao")
and the per-token stopping criterion ("Computacao Dinamica").

Pins used: hand-worked values (tests/golden), brute force of the objective on tiny inputs
(explicit zeta products, least squares by SVD), the closed form of one CG step, the
Cholesky solve after d_k CG steps, ridge regression (gamma = 1, Lambda = lambda I),
Sherman-Morrison (gamma = 0), symmetry and positive definiteness, and the minimality of
the dynamic iteration count measured with the true residual.
"""
import json
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.optimize

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_examples.json")


def _zeta(gamma, t, tp):
    """zeta_{t t'} = prod_{s=t'+1..t} gamma_s (0-based token indices), by explicit product."""
    z = 1.0
    for s in range(tp + 1, t + 1):
        z *= gamma[s]
    return z


def _explicit_states(k, v, gamma, t):
    """H_t, G_t from the definition as sums of zeta-weighted outer products (no recurrence)."""
    dk, dv = k.shape[1], v.shape[1]
    H = np.zeros((dk, dk))
    G = np.zeros((dv, dk))
    for tp in range(t + 1):
        z = _zeta(gamma, t, tp)
        H += z * np.outer(k[tp], k[tp])
        G += z * np.outer(v[tp], k[tp])
    return H, G


def _objective(Phi, k, v, gamma, lam, t):
    """The Mesa objective at token t, evaluated straight from its definition."""
    loss = 0.0
    for tp in range(t + 1):
        e = v[tp] - Phi @ k[tp]
        loss += 0.5 * _zeta(gamma, t, tp) * float(e @ e)
    return loss + 0.5 * float(np.trace(Phi @ np.diag(lam) @ Phi.T))


def _rand_case(rng, T, dk, dv, gamma_lo=0.5, gamma_hi=1.0):
    k = rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    q = rng.standard_normal((T, dk))
    gamma = rng.uniform(gamma_lo, gamma_hi, T)
    lam = rng.uniform(0.3, 1.5, dk)
    return q, k, v, gamma, lam


def _fwd1(q, k, v, gamma, lam, cg_iters, cg_tol=0.0, lib=None):
    """Oracle forward on a single (batch, head) unit."""
    out, it = oracle.forward(q[None, None], k[None, None], v[None, None], gamma[None, None],
                             lam[None], cg_iters, cg_tol, lib=lib)
    return out[0, 0], it[0, 0]


# --------------------------------------------------------------------------------------
# hand-worked values


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_worked_examples(case):
    arr = lambda key: np.array(case[key], dtype=np.float64)
    out, it = _fwd1(arr("q"), arr("k"), arr("v"), arr("gamma"), arr("lam"), case["cg_iters"])
    np.testing.assert_allclose(out, arr("out"), rtol=1e-13, atol=1e-14)
    assert (it == case["cg_iters"]).all()


# --------------------------------------------------------------------------------------
# states and the objective


def test_states_match_explicit_zeta_products():
    rng = np.random.default_rng(1)
    T, dk, dv = 7, 3, 2
    _, k, v, gamma, _ = _rand_case(rng, T, dk, dv)
    gamma[2] = 0.0
    gamma[4] = 1.0
    Ha, Ga = oracle.state_trace(k, v, gamma)
    for t in range(T):
        H, G = _explicit_states(k, v, gamma, t)
        np.testing.assert_allclose(Ha[t], H, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(Ga[t], G, rtol=1e-13, atol=1e-14)


def test_states_symmetric_and_shifted_pd():
    rng = np.random.default_rng(2)
    q, k, v, gamma, lam = _rand_case(rng, 40, 5, 3)
    Ha, _ = oracle.state_trace(k, v, gamma)
    for t in range(40):
        assert np.array_equal(Ha[t], Ha[t].T)
        ev = np.linalg.eigvalsh(Ha[t] + np.diag(lam))
        assert ev.min() >= lam.min() * (1 - 1e-12)


@pytest.mark.parametrize("seed", [3, 4])
def test_output_is_minimiser_of_objective_least_squares(seed):
    """Brute force: minimise the objective as a weighted ridge least-squares problem by SVD
    (np.linalg.lstsq on the stacked system), independent of H/G and of CG."""
    rng = np.random.default_rng(seed)
    T, dk, dv = 6, 4, 3
    q, k, v, gamma, lam = _rand_case(rng, T, dk, dv)
    out, _ = _fwd1(q, k, v, gamma, lam, cg_iters=dk)
    for t in range(T):
        w = np.sqrt([_zeta(gamma, t, tp) for tp in range(t + 1)])
        # rows: sqrt(zeta) k_t'^T Phi^T = sqrt(zeta) v_t'^T ; sqrt(Lambda) Phi^T = 0
        A = np.vstack([w[:, None] * k[: t + 1], np.diag(np.sqrt(lam))])
        Bm = np.vstack([w[:, None] * v[: t + 1], np.zeros((dk, dv))])
        PhiT = np.linalg.lstsq(A, Bm, rcond=None)[0]
        np.testing.assert_allclose(out[t], PhiT.T @ q[t], rtol=1e-9, atol=1e-10)


def test_objective_gradient_vanishes_and_perturbations_increase():
    """At the oracle's Phi (recovered column by column from its outputs with q = e_j) the
    objective's finite-difference gradient is zero and random perturbations increase it."""
    rng = np.random.default_rng(5)
    T, dk, dv = 5, 3, 2
    _, k, v, gamma, lam = _rand_case(rng, T, dk, dv)
    t = T - 1
    Phi = np.zeros((dv, dk))
    for j in range(dk):
        qj = np.zeros((T, dk))
        qj[:, j] = 1.0
        out, _ = _fwd1(qj, k, v, gamma, lam, cg_iters=dk)
        Phi[:, j] = out[t]
    f0 = _objective(Phi, k, v, gamma, lam, t)
    h = 1e-6
    grad = np.zeros_like(Phi)
    for idx in np.ndindex(Phi.shape):
        E = np.zeros_like(Phi)
        E[idx] = h
        grad[idx] = (_objective(Phi + E, k, v, gamma, lam, t) - _objective(Phi - E, k, v, gamma, lam, t)) / (2 * h)
    assert np.abs(grad).max() < 1e-7
    for _ in range(20):
        assert _objective(Phi + 1e-3 * rng.standard_normal(Phi.shape), k, v, gamma, lam, t) > f0
    # and a general-purpose optimiser started elsewhere lands on the same Phi
    res = scipy.optimize.minimize(lambda x: _objective(x.reshape(dv, dk), k, v, gamma, lam, t),
                                  np.zeros(dv * dk), method="BFGS", options={"gtol": 1e-12})
    np.testing.assert_allclose(res.x.reshape(dv, dk), Phi, atol=1e-6)


# --------------------------------------------------------------------------------------
# conjugate gradient


def test_one_cg_step_closed_form():
    """One CG step from x0 = 0 is the exact line search along q: x1 = (q.q / q.Aq) q."""
    rng = np.random.default_rng(6)
    T, dk, dv = 9, 6, 4
    q, k, v, gamma, lam = _rand_case(rng, T, dk, dv)
    out, it = _fwd1(q, k, v, gamma, lam, cg_iters=1)
    assert (it == 1).all()
    for t in range(T):
        H, G = _explicit_states(k, v, gamma, t)
        A = H + np.diag(lam)
        x1 = (q[t] @ q[t]) / (q[t] @ A @ q[t]) * q[t]
        np.testing.assert_allclose(out[t], G @ x1, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dk", [2, 5, 8, 16])
def test_dk_cg_steps_reach_cholesky_solve(dk):
    rng = np.random.default_rng(7 + dk)
    T, dv = 12, 3
    q, k, v, gamma, lam = _rand_case(rng, T, dk, dv, 0.7, 1.0)
    k /= np.linalg.norm(k, axis=1, keepdims=True)  # unit keys, as in every workload
    lam += 0.5  # well conditioned: exact-arithmetic termination shows through fp64
    out, it = _fwd1(q, k, v, gamma, lam, cg_iters=dk)
    for t in range(T):
        H, G = _explicit_states(k, v, gamma, t)
        xs = scipy.linalg.cho_solve(scipy.linalg.cho_factor(H + np.diag(lam)), q[t])
        ref = G @ xs
        # CG in fp64 after d_k steps: round-off grows with the condition number
        assert np.linalg.norm(out[t] - ref) <= 1e-8 * np.linalg.norm(ref)


def test_cg_residual_decreases_to_exact_on_dense_system():
    """Standalone CG routine: the true residual after n steps of an n x n SPD system is at
    round-off level, and the A-norm of the error decreases monotonically (a property of CG)."""
    rng = np.random.default_rng(8)
    n = 10
    M = rng.standard_normal((n, n))
    Hm = M @ M.T / n
    lam = rng.uniform(0.5, 1.0, n)
    A = Hm + np.diag(lam)
    b = rng.standard_normal(n)
    xs = np.linalg.solve(A, b)
    prev = np.inf
    for kk in range(n + 1):
        x, it = oracle.cg(Hm, lam, b, kk)
        assert it == kk
        e = x - xs
        en = float(e @ A @ e)
        assert en <= prev * (1 + 1e-12) + 1e-28
        prev = en
    assert np.linalg.norm(b - A @ x) < 1e-10 * np.linalg.norm(b)


def test_ridge_regression_special_case():
    """gamma = 1 and Lambda = lambda I: o_t = V^T K (K^T K + lambda I)^-1 q_t (numpy solve)."""
    rng = np.random.default_rng(9)
    T, dk, dv, lamv = 10, 4, 3, 0.7
    q, k, v, _, _ = _rand_case(rng, T, dk, dv)
    gamma = np.ones(T)
    lam = np.full(dk, lamv)
    out, _ = _fwd1(q, k, v, gamma, lam, cg_iters=dk)
    for t in range(T):
        K, V = k[: t + 1], v[: t + 1]
        ref = V.T @ K @ np.linalg.solve(K.T @ K + lamv * np.eye(dk), q[t])
        np.testing.assert_allclose(out[t], ref, rtol=1e-9, atol=1e-10)


def test_sherman_morrison_special_case():
    """gamma = 0 keeps only the current token: o_t = v_t (k^T L^-1 q) / (1 + k^T L^-1 k)."""
    rng = np.random.default_rng(10)
    T, dk, dv = 6, 5, 3
    q, k, v, _, lam = _rand_case(rng, T, dk, dv)
    gamma = np.zeros(T)
    out, _ = _fwd1(q, k, v, gamma, lam, cg_iters=dk)
    for t in range(T):
        ref = v[t] * (k[t] @ (q[t] / lam)) / (1.0 + k[t] @ (k[t] / lam))
        np.testing.assert_allclose(out[t], ref, rtol=1e-9, atol=1e-10)


def test_dynamic_stop_is_first_iterate_meeting_true_residual():
    """Dynamic mode stops at the first k with ||q - A x_k|| <= tol ||q||; checked with the
    true residual of fixed-count runs (replay), computed here from explicit states."""
    rng = np.random.default_rng(11)
    T, dk, dv, tol = 30, 8, 2, 1e-3
    q, k, v, gamma, lam = _rand_case(rng, T, dk, dv, 0.8, 1.0)
    lam *= 0.2
    out, it = _fwd1(q, k, v, gamma, lam, cg_iters=50, cg_tol=tol)
    assert it.min() >= 1 and it.max() <= 50
    for t in range(T):
        H, _ = _explicit_states(k, v, gamma, t)
        A = H + np.diag(lam)
        n = int(it[t])
        x_n, _ = oracle.cg(H, lam, q[t], n)
        assert np.linalg.norm(q[t] - A @ x_n) <= tol * np.linalg.norm(q[t]) * (1 + 1e-6)
        x_m, _ = oracle.cg(H, lam, q[t], n - 1)
        assert np.linalg.norm(q[t] - A @ x_m) > tol * np.linalg.norm(q[t]) * (1 - 1e-6)


def test_replay_reproduces_dynamic_run():
    rng = np.random.default_rng(12)
    q, k, v, gamma, lam = _rand_case(rng, 25, 6, 4)
    out, it = _fwd1(q, k, v, gamma, lam, cg_iters=40, cg_tol=1e-4)
    o2, it2 = oracle.forward(q[None, None], k[None, None], v[None, None], gamma[None, None], lam[None],
                             0, 0.0, replay=it[None, None])
    assert np.array_equal(it, it2[0, 0])
    np.testing.assert_array_equal(out, o2[0, 0])


def test_zero_query_edge_cases():
    rng = np.random.default_rng(13)
    q, k, v, gamma, lam = _rand_case(rng, 5, 4, 3)
    q[2] = 0.0
    out, it = _fwd1(q, k, v, gamma, lam, cg_iters=7, cg_tol=1e-3)
    assert it[2] == 0 and np.all(out[2] == 0)
    out, it = _fwd1(q, k, v, gamma, lam, cg_iters=7, cg_tol=0.0)
    assert it[2] == 7 and np.all(out[2] == 0)
    assert (it == 7).all()


def test_decode_steps_equal_forward():
    """T decode steps from a zero state give the forward outputs and the final states."""
    rng = np.random.default_rng(14)
    N, heads, T, dk, dv = 2, 3, 9, 5, 4
    q = rng.standard_normal((N, heads, T, dk))
    k = rng.standard_normal((N, heads, T, dk))
    v = rng.standard_normal((N, heads, T, dv))
    gamma = rng.uniform(0.5, 1.0, (N, heads, T))
    lam = rng.uniform(0.3, 1.0, (heads, dk))
    out, it, Hf, Gf = oracle.forward(q, k, v, gamma, lam, 6, 1e-5, want_final=True)
    Hs = np.zeros((N, heads, dk, dk))
    Gs = np.zeros((N, heads, dv, dk))
    for t in range(T):
        o, i = oracle.decode_step(Hs, Gs, q[:, :, t], k[:, :, t], v[:, :, t], gamma[:, :, t], lam, 6, 1e-5)
        np.testing.assert_array_equal(o, out[:, :, t])
        np.testing.assert_array_equal(i, it[:, :, t])
    np.testing.assert_array_equal(Hs, Hf)
    np.testing.assert_array_equal(Gs, Gf)


def test_initial_state_continues_the_sequence():
    """Forward over T1 then forward over T2 from the exported state = forward over T1+T2."""
    rng = np.random.default_rng(15)
    T, dk, dv = 16, 4, 3
    q, k, v, gamma, lam = _rand_case(rng, T, dk, dv)
    a = lambda x: x[None, None]
    out, it = oracle.forward(a(q), a(k), a(v), a(gamma), lam[None], 4)
    o1, _, Hf, Gf = oracle.forward(a(q[:7]), a(k[:7]), a(v[:7]), a(gamma[:7]), lam[None], 4, want_final=True)
    o2, _ = oracle.forward(a(q[7:]), a(k[7:]), a(v[7:]), a(gamma[7:]), lam[None], 4, H0=Hf, G0=Gf)
    np.testing.assert_array_equal(np.concatenate([o1, o2], axis=2), out)


def test_heads_use_their_own_lambda_and_units_are_independent():
    rng = np.random.default_rng(16)
    B, heads, T, dk, dv = 2, 3, 6, 4, 2
    q = rng.standard_normal((B, heads, T, dk))
    k = rng.standard_normal((B, heads, T, dk))
    v = rng.standard_normal((B, heads, T, dv))
    gamma = rng.uniform(0.5, 1.0, (B, heads, T))
    lam = rng.uniform(0.3, 1.0, (heads, dk))
    out, _ = oracle.forward(q, k, v, gamma, lam, dk)
    for b in range(B):
        for h in range(heads):
            o1, _ = _fwd1(q[b, h], k[b, h], v[b, h], gamma[b, h], lam[h], dk)
            np.testing.assert_array_equal(out[b, h], o1)


def test_readout_magnitude_one_token_closed_form():
    """The readout magnitude s_t = || |G_t| |x_t| || the oracle reports next to o_t, pinned
    on one token after one CG step: H = k k^T, G = v k^T and x_1 = c q with
    c = q.q / q.(H + Lambda) q > 0, so |G| |x| = |v| (|k| . |x|) and s = ||v|| c sum_b |k_b q_b|."""
    rng = np.random.default_rng(31)
    dk, dv = 5, 3
    q, k, v = rng.standard_normal(dk), rng.standard_normal(dk), rng.standard_normal(dv)
    lam = rng.uniform(0.3, 1.0, dk)
    c = (q @ q) / (q @ (np.outer(k, k) @ q + lam * q))
    a = lambda x: np.asarray(x, dtype=np.float64)[None, None, None]
    s = np.zeros((1, 1, 1))
    o, _ = oracle.forward(a(q), a(k), a(v), a([0.7]).reshape(1, 1, 1), lam[None], 1, scale_out=s)
    np.testing.assert_allclose(o[0, 0, 0], v * c * (k @ q), rtol=1e-12)
    np.testing.assert_allclose(s[0, 0, 0], np.linalg.norm(v) * c * np.abs(k * q).sum(), rtol=1e-12)


def test_readout_magnitude_properties():
    """s_t >= ||o_t|| on every token (equality in one dimension); flipping the values' sign
    flips o and keeps s; scaling the values scales both; the decode step reports the same
    magnitudes as the forward."""
    rng = np.random.default_rng(32)
    T, dk, dv = 40, 6, 4
    q, k, v, gamma, lam = _rand_case(rng, T, dk, dv)
    a = lambda x: x[None, None]
    s = np.zeros((1, 1, T))
    o, _ = oracle.forward(a(q), a(k), a(v), a(gamma), lam[None], 3, scale_out=s)
    n = np.linalg.norm(o[0, 0], axis=-1)
    assert np.all(s[0, 0] >= n * (1 - 1e-12)) and np.any(s[0, 0] > n * 1.01)
    s2 = np.zeros((1, 1, T))
    o2, _ = oracle.forward(a(q), a(k), a(-2.0 * v), a(gamma), lam[None], 3, scale_out=s2)
    np.testing.assert_allclose(o2, -2.0 * o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(s2, 2.0 * s, rtol=1e-12)
    s1 = np.zeros((1, 1, T))
    o1, _ = oracle.forward(a(q[:, :1]), a(k[:, :1]), a(v[:, :1]), a(gamma), lam[None, :1], 2, scale_out=s1)
    np.testing.assert_allclose(s1[0, 0], np.abs(o1[0, 0, :, 0]), rtol=1e-12)
    Hs, Gs = np.zeros((1, 1, dk, dk)), np.zeros((1, 1, dv, dk))
    for t in range(T):
        sd = np.zeros((1, 1))
        oracle.decode_step(Hs, Gs, q[t][None, None], k[t][None, None], v[t][None, None], gamma[t].reshape(1, 1),
                           lam[None], 3, scale_out=sd)
        assert sd[0, 0] == s[0, 0, t]
