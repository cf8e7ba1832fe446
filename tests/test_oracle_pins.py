"""Pins for the fp64 oracle: each test checks it against something other than itself.

Sources (gist.science summary of arXiv 2512.12602, "Exact Flow Linear
Attention: Exact Solution from Continuous-Time Dynamics"):
  ODE              page es, Metodologia item 1
  closed form      page es, Metodologia item 2
  update rule, alpha   page es, Metodologia item 3
  Euler/delta rule page es, Contribuciones Clave item 1 (delta rule = explicit Euler step)
  key contraction  page es, Contribuciones Clave item 4 (factor e^{-beta lambda})
  WY/UT chunking   page es, Metodologia item 3, last paragraph
"""
import math

import numpy as np
import pytest
import scipy.linalg

import oracle

RNG = np.random.default_rng(1234)


def _rand_k(d, norm):
    k = RNG.standard_normal(d)
    return k / np.linalg.norm(k) * norm


# ----------------------------------------------------------------- P1 closed form
@pytest.mark.parametrize("x", [1e-9, 1e-6, 1e-3, 0.05, 0.3, 1.0, 4.0, 30.0, 100.0])
@pytest.mark.parametrize("d", [1, 3, 6])
def test_p1_closed_form_matches_matrix_exponential(x, d):
    """I - alpha k k^T equals expm(-beta k k^T): scipy's Pade expm and an eigendecomposition."""
    lam = RNG.uniform(0.2, 5.0)
    beta = x / lam
    k = _rand_k(d, math.sqrt(lam))
    A = np.outer(k, k)
    closed = np.eye(d) - oracle.alpha(beta, lam) * A
    ref_pade = scipy.linalg.expm(-beta * A)
    w, V = np.linalg.eigh(A)
    ref_eig = (V * np.exp(-beta * w)) @ V.T
    assert np.max(np.abs(closed - ref_pade)) < 1e-12
    assert np.max(np.abs(closed - ref_eig)) < 1e-12


def test_p1_rank1_power_identity_and_series():
    """A^n = lambda^{n-1} A (page es item 2), and the Taylor series of exp(-beta A) summed
    term by term (with scaling and squaring) reproduces the closed form."""
    d = 5
    k = RNG.standard_normal(d)
    lam = float(k @ k)
    A = np.outer(k, k)
    P = A.copy()
    for n in range(2, 7):
        P = P @ A
        assert np.allclose(P, lam ** (n - 1) * A, rtol=1e-12, atol=0)
    beta = 3.0 / lam
    s = 6
    M = -beta * A / 2 ** s
    E = np.eye(d)
    term = np.eye(d)
    for n in range(1, 30):
        term = term @ M / n
        E = E + term
    for _ in range(s):
        E = E @ E
    assert np.max(np.abs(E - (np.eye(d) - oracle.alpha(beta, lam) * A))) < 1e-12


# -------------------------------------------------------------- P2 ODE flow
def _rk4(S0, k, v, beta, n):
    A = np.outer(k, k)
    b = np.outer(k, v)
    f = lambda S: -A @ S + b  # noqa: E731
    h = beta / n
    S = S0.copy()
    for _ in range(n):
        k1 = f(S)
        k2 = f(S + 0.5 * h * k1)
        k3 = f(S + 0.5 * h * k2)
        k4 = f(S + h * k3)
        S = S + (h / 6.0) * (k1 + 2 * k2 + 2 * k3 + k4)
    return S


@pytest.mark.parametrize("x", [1e-4, 0.5, 3.0, 20.0, 100.0])
def test_p2_one_step_is_the_exact_ode_flow(x):
    """One oracle step equals (a) fine RK4 integration of dS/dt = -kk^T S + kv^T over a
    ZOH interval of length beta and (b) the Van Loan block exponential of the same ODE."""
    dk, dv = 4, 3
    lam = RNG.uniform(0.5, 4.0)
    beta = x / lam
    k = _rand_k(dk, math.sqrt(lam))
    v = RNG.standard_normal(dv)
    q = RNG.standard_normal(dk)
    S0 = RNG.standard_normal((dk, dv))
    _, Sn = oracle.step(q[None, None], k[None, None], v[None, None],
                        np.array([[beta]]), S0[None, None])
    Sn = Sn[0, 0]
    n = int(20 * x) + 1000
    assert np.max(np.abs(Sn - _rk4(S0, k, v, beta, n))) < 1e-10
    # Van Loan: d/dt [S; I] with generator [[-A, b], [0, 0]]
    Mg = np.zeros((dk + dv, dk + dv))
    Mg[:dk, :dk] = -np.outer(k, k)
    Mg[:dk, dk:] = np.outer(k, v)
    E = scipy.linalg.expm(beta * Mg)
    exact = E[:dk, :dk] @ S0 + E[:dk, dk:]
    assert np.max(np.abs(Sn - exact)) < 1e-12


# ----------------------------------------------------- P3 key-direction contraction
@pytest.mark.parametrize("x", [1e-5, 0.7, 5.0, 60.0])
def test_p3_key_direction_contraction(x):
    dk, dv = 6, 4
    lam = RNG.uniform(0.5, 4.0)
    beta = x / lam
    k = _rand_k(dk, math.sqrt(lam))
    v = RNG.standard_normal(dv)
    S0 = RNG.standard_normal((dk, dv))
    _, Sn = oracle.step(np.zeros((1, 1, dk)), k[None, None], v[None, None],
                        np.array([[beta]]), S0[None, None])
    Sn = Sn[0, 0]
    khat = k / np.linalg.norm(k)
    e = math.exp(-x)
    # along k: contracted by e^{-beta lambda} towards v^T (scaled by ||k||)
    lhs = khat @ Sn
    rhs = e * (khat @ S0) + (1 - e) * v / np.linalg.norm(k)
    assert np.max(np.abs(lhs - rhs)) < 1e-12 * (1 + np.max(np.abs(rhs)))
    # orthogonal to k: untouched
    P = np.eye(dk) - np.outer(khat, khat)
    assert np.max(np.abs(P @ Sn - P @ S0)) < 1e-12


def test_p3_stiff_limit_replaces_key_direction():
    dk, dv = 5, 3
    k = _rand_k(dk, 3.0)
    v = RNG.standard_normal(dv)
    S0 = RNG.standard_normal((dk, dv))
    _, Sn = oracle.step(np.zeros((1, 1, dk)), k[None, None], v[None, None],
                        np.array([[500.0]]), S0[None, None])
    assert np.max(np.abs(k @ Sn[0, 0] - v)) < 1e-12
    assert abs(oracle.alpha(500.0, 9.0) * 9.0 - 1.0) < 1e-15


# --------------------------------------------------------------- alpha limits
def test_alpha_limits_and_high_precision_values():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    for beta, lam in [(0.3, 1e-300), (0.7, 1e-20), (0.5, 1e-9), (0.9, 1e-3), (0.2, 0.3),
                      (0.6, 7.0), (0.95, 100.0), (2.0, 400.0), (-0.3, 2.0)]:
        ref = -mp.expm1(-mp.mpf(beta) * mp.mpf(lam)) / mp.mpf(lam)
        got = oracle.alpha(beta, lam)
        assert abs(got - float(ref)) <= 4e-16 * abs(float(ref)), (beta, lam)
    assert oracle.alpha(0.37, 0.0) == 0.37          # lambda = 0: alpha = beta
    assert oracle.alpha(0.0, 5.0) == 0.0
    assert oracle.alpha(0.37, 2.0, euler=True) == 0.37


def test_alpha_derivatives_against_high_precision():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    f = lambda b, l: (1 - mp.exp(-b * l)) / l  # noqa: E731
    for beta, lam in [(0.5, 1e-7), (0.5, 0.02), (0.5, 0.0999), (0.5, 0.1001), (0.8, 0.3),
                      (0.3, 5.0), (0.9, 60.0)]:
        b, l = mp.mpf(beta), mp.mpf(lam)
        dl = mp.diff(lambda z: f(b, z), l)
        db = mp.diff(lambda z: f(z, l), b)
        assert abs(oracle.dalpha_dlambda(beta, lam) - float(dl)) <= 1e-13 * abs(float(dl))
        assert abs(oracle.dalpha_dbeta(beta, lam) - float(db)) <= 1e-14 * abs(float(db))


# --------------------------------------------------------------- P4/P5 Euler
def test_p4_euler_mode_is_explicit_euler_step_of_the_ode():
    B, H, L, dk, dv = 1, 2, 9, 4, 3
    q = RNG.standard_normal((B, H, L, dk))
    k = RNG.standard_normal((B, H, L, dk))
    v = RNG.standard_normal((B, H, L, dv))
    beta = RNG.uniform(0.05, 0.9, (B, H, L))
    S0 = RNG.standard_normal((B, H, dk, dv))
    o, Sf = oracle.fwd(q, k, v, beta, S0, euler=True)
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy()
            for t in range(L):
                kk, vv = k[b, h, t], v[b, h, t]
                S = S + beta[b, h, t] * (-np.outer(kk, kk) @ S + np.outer(kk, vv))
                assert np.allclose(o[b, h, t], S.T @ q[b, h, t], rtol=0, atol=1e-12)
            assert np.allclose(Sf[b, h], S, rtol=0, atol=1e-12)


def test_p5_unit_keys_exact_flow_equals_delta_rule_with_rescaled_beta():
    B, H, L, dk, dv = 1, 1, 20, 5, 4
    q = RNG.standard_normal((B, H, L, dk))
    k = RNG.standard_normal((B, H, L, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = RNG.standard_normal((B, H, L, dv))
    beta = RNG.uniform(0.1, 3.0, (B, H, L))
    o1, S1 = oracle.fwd(q, k, v, beta)
    o2, S2 = oracle.fwd(q, k, v, 1 - np.exp(-beta), euler=True)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(S1 - S2)) < 1e-12


def test_scalar_state_closed_form():
    """d_k = d_v = 1: S_t = e^{-beta k^2} S_{t-1} + (1 - e^{-beta k^2}) v / k exactly."""
    L = 40
    k = RNG.uniform(0.1, 3.0, L) * RNG.choice([-1, 1], L)
    v = RNG.standard_normal(L)
    q = RNG.standard_normal(L)
    beta = RNG.uniform(0.01, 2.0, L)
    o, Sf = oracle.fwd(q.reshape(1, 1, L, 1), k.reshape(1, 1, L, 1), v.reshape(1, 1, L, 1),
                       beta.reshape(1, 1, L), np.full((1, 1, 1, 1), 0.25))
    S = 0.25
    for t in range(L):
        e = math.exp(-beta[t] * k[t] ** 2)
        S = e * S + (1 - e) * v[t] / k[t]
        assert abs(o[0, 0, t, 0] - S * q[t]) < 1e-13
    assert abs(Sf[0, 0, 0, 0] - S) < 1e-13


# ------------------------------------------------------------- P6 chunked = recurrent
def _chunked_ut(q, k, v, beta, S0, C):
    """Brute-force chunkwise WY/UT evaluation with a dense inverse (numpy fp64)."""
    B, H, L, dk = k.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, L, dv))
    Sf = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy()
            for c0 in range(0, L, C):
                K = k[b, h, c0:c0 + C]
                V = v[b, h, c0:c0 + C]
                Q = q[b, h, c0:c0 + C]
                lam = np.sum(K * K, axis=1)
                a = (1 - np.exp(-beta[b, h, c0:c0 + C] * lam)) / lam
                n = K.shape[0]
                Amat = np.tril(a[:, None] * (K @ K.T), -1)
                T = np.linalg.inv(np.eye(n) + Amat)
                W = T @ (a[:, None] * K)
                U = T @ (a[:, None] * V)
                Up = U - W @ S
                o[b, h, c0:c0 + C] = Q @ S + np.tril(Q @ K.T) @ Up
                S = S + K.T @ Up
            Sf[b, h] = S
    return o, Sf


@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_p6_chunked_ut_equals_recurrence(C):
    B, H, L, dk, dv = 1, 2, 50, 8, 6      # L = 50: ragged tail for C = 4, 16
    q = RNG.standard_normal((B, H, L, dk))
    k = RNG.standard_normal((B, H, L, dk)) * RNG.uniform(0.2, 2.0, (B, H, L, 1))
    v = RNG.standard_normal((B, H, L, dv))
    beta = RNG.uniform(0.05, 0.95, (B, H, L))
    S0 = 0.1 * RNG.standard_normal((B, H, dk, dv))
    o1, S1 = oracle.fwd(q, k, v, beta, S0)
    o2, S2 = _chunked_ut(q, k, v, beta, S0, C)
    assert np.max(np.abs(o1 - o2)) < 1e-10
    assert np.max(np.abs(S1 - S2)) < 1e-10


def test_resume_chaining():
    B, H, L1, L2, dk, dv = 1, 2, 13, 17, 4, 5
    q = RNG.standard_normal((B, H, L1 + L2, dk))
    k = RNG.standard_normal((B, H, L1 + L2, dk))
    v = RNG.standard_normal((B, H, L1 + L2, dv))
    beta = RNG.uniform(0, 1, (B, H, L1 + L2))
    o, Sf = oracle.fwd(q, k, v, beta)
    oa, Sa = oracle.fwd(q[:, :, :L1], k[:, :, :L1], v[:, :, :L1], beta[:, :, :L1])
    ob, Sb = oracle.fwd(q[:, :, L1:], k[:, :, L1:], v[:, :, L1:], beta[:, :, L1:], Sa)
    assert np.max(np.abs(np.concatenate([oa, ob], 2) - o)) < 1e-13
    assert np.max(np.abs(Sb - Sf)) < 1e-13


# ------------------------------------------------------------------ P7 backward
@pytest.mark.parametrize("euler", [False, True])
def test_p7_backward_matches_central_differences(euler):
    """Every input of a tiny case (L = 70 crosses the oracle's 64-token checkpoint)."""
    B, H, L, dk, dv = 1, 1, 70, 3, 2
    rng = np.random.default_rng(7)
    q = rng.standard_normal((B, H, L, dk))
    k = rng.standard_normal((B, H, L, dk)) * rng.uniform(0.3, 2.0, (B, H, L, 1))
    v = rng.standard_normal((B, H, L, dv))
    beta = rng.uniform(0.05, 0.95, (B, H, L))
    S0 = 0.3 * rng.standard_normal((B, H, dk, dv))
    dO = rng.standard_normal((B, H, L, dv))
    dSf = rng.standard_normal((B, H, dk, dv))

    def loss(q_, k_, v_, b_, s_):
        o, Sf = oracle.fwd(q_, k_, v_, b_, s_, euler=euler)
        return float(np.sum(o * dO) + np.sum(Sf * dSf))

    grads = oracle.bwd(q, k, v, beta, dO, S0, dSf, euler=euler)
    args = [q, k, v, beta, S0]
    h = 1e-6
    for idx, (x, g) in enumerate(zip(args, grads)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            m = it.multi_index
            xp = [a.copy() for a in args]
            xm = [a.copy() for a in args]
            xp[idx][m] += h
            xm[idx][m] -= h
            fd[m] = (loss(*xp) - loss(*xm)) / (2 * h)
        err = np.max(np.abs(fd - g)) / max(1.0, np.max(np.abs(fd)))
        assert err < 1e-6, (idx, err)


def test_p7_no_upstream_state_grad_and_zero_s0():
    """dS_final = None and S0 = None are the zero tensors."""
    B, H, L, dk, dv = 1, 1, 10, 3, 3
    q = RNG.standard_normal((B, H, L, dk))
    k = RNG.standard_normal((B, H, L, dk))
    v = RNG.standard_normal((B, H, L, dv))
    beta = RNG.uniform(0, 1, (B, H, L))
    dO = RNG.standard_normal((B, H, L, dv))
    g1 = oracle.bwd(q, k, v, beta, dO)
    g2 = oracle.bwd(q, k, v, beta, dO, np.zeros((B, H, dk, dv)), np.zeros((B, H, dk, dv)))
    for a, b in zip(g1, g2):
        assert np.array_equal(a, b)
