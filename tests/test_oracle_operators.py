"""Pins of the oracle's expansion operators (P2M, M2M, M2L, L2L, L2P, D^n).

Each operator is checked against something other than itself: symbolic
derivatives (sympy), closed forms, exact polynomial identities, the page's
printed monopole/dipole formulas (JZ-FMM page, "Calculating a node-node
interaction") and the direct sum.
"""
import math

import numpy as np
import pytest
import sympy as sp

import oracle


def mono(x, n):
    return x[0] ** n[0] * x[1] ** n[1] * x[2] ** n[2] / (
        math.factorial(n[0]) * math.factorial(n[1]) * math.factorial(n[2]))


def test_coefficient_order():
    """Graded order; within a degree nx descending, then ny descending."""
    seen = []
    for d in range(7):
        for nx in range(d, -1, -1):
            for ny in range(d - nx, -1, -1):
                seen.append(oracle.mindex(nx, ny, d - nx - ny))
    assert seen == list(range(oracle.ncoef(6)))
    assert [oracle.ncoef(p) for p in range(2, 7)] == [10, 20, 35, 56, 84]


def test_derivatives_match_symbolic():
    """D^n(R) = d^n(1/r) against sympy's exact derivatives, |n| <= 8."""
    p = 8
    x, y, z = sp.symbols("x y z", real=True)
    f = 1 / sp.sqrt(x * x + y * y + z * z)
    R = (0.37, -1.21, 0.83)
    mi = oracle.multi_indices(p)
    cache = {(0, 0, 0): f}

    def deriv(n):
        n = tuple(int(v) for v in n)
        if n not in cache:
            i = 0 if n[0] > 0 else (1 if n[1] > 0 else 2)
            m = list(n)
            m[i] -= 1
            cache[n] = sp.diff(deriv(m), (x, y, z)[i])
        return cache[n]

    want = np.array([float(deriv(n).subs({x: R[0], y: R[1], z: R[2]})) for n in mi])
    got = oracle.derivs(p, R)
    order = mi.sum(axis=1)
    # rounding of the recurrence grows like l! r^-(l+1)
    scale = np.abs(want) + np.array([math.factorial(l) for l in order]) * np.linalg.norm(R) ** -(order + 1.0)
    assert np.max(np.abs(got - want) / scale) < 1e-13


def test_derivatives_are_harmonic():
    """1/r is harmonic: D^{n+2ex} + D^{n+2ey} + D^{n+2ez} = 0."""
    p = 10
    D = oracle.derivs(p, [0.5, 0.9, -0.4])
    mi = oracle.multi_indices(p - 2)
    r = np.linalg.norm([0.5, 0.9, -0.4])
    for n in mi:
        s = sum(D[oracle.mindex(*(n + 2 * np.eye(3, dtype=int)[a]))] for a in range(3))
        assert abs(s) < 1e-12 * r ** -(n.sum() + 3) * math.factorial(n.sum() + 2)


def test_p2m_single_particle_closed_form():
    """One particle of mass m at offset s: M_n = m s^n / n!."""
    p = 6
    c = np.array([0.1, 0.2, 0.3])
    s = np.array([0.05, -0.02, 0.07])
    M = oracle.p2m(p, (c + s)[None, :], [1.7], c)
    mi = oracle.multi_indices(p)
    np.testing.assert_allclose(M, [1.7 * mono(s, n) for n in mi], rtol=1e-14, atol=1e-300)


def test_p2m_page_low_moments():
    """Total mass, dipole and second moment of the page's moment equations."""
    rng = np.random.default_rng(1)
    x = rng.random((40, 3))
    m = rng.uniform(0.5, 1.5, 40)
    c = np.array([0.4, 0.5, 0.6])
    M = oracle.p2m(2, x, m, c)
    s = x - c
    assert abs(M[0] - m.sum()) < 1e-14 * m.sum()
    for a in range(3):
        e = [0, 0, 0]
        e[a] = 1
        np.testing.assert_allclose(M[oracle.mindex(*e)], np.sum(m * s[:, a]), rtol=1e-13)
        for b in range(3):
            e2 = [0, 0, 0]
            e2[a] += 1
            e2[b] += 1
            second = np.sum(m * s[:, a] * s[:, b])  # M^(2)_{ab} of the page
            fact = 2.0 if a == b else 1.0  # n! normalisation of the stored coefficient
            np.testing.assert_allclose(M[oracle.mindex(*e2)] * fact, second, rtol=1e-12)


@pytest.mark.parametrize("p", [2, 4, 6])
def test_m2m_equals_direct_p2m(p):
    """Moments translated from children equal moments taken about the parent."""
    rng = np.random.default_rng(p)
    parts = [rng.random((30, 3)) * 0.3 + o for o in ([0, 0, 0], [0.5, 0.1, 0.2], [0.2, 0.6, 0.5])]
    masses = [rng.uniform(0.1, 1.0, 30) for _ in parts]
    cp = np.array([0.45, 0.4, 0.35])
    Mp = np.zeros(oracle.ncoef(p))
    for x, m in zip(parts, masses):
        cc = x.mean(axis=0)
        Mp += oracle.m2m(p, oracle.p2m(p, x, m, cc), cc - cp)
    want = oracle.p2m(p, np.vstack(parts), np.concatenate(masses), cp)
    np.testing.assert_allclose(Mp, want, rtol=1e-12, atol=1e-14 * np.abs(want).max())


def test_m2l_low_order_terms_are_the_page_formulas():
    """p = 1: Phi_B(c_A) = -G[M/R + M1.R/R^3], grad = G[M R/R^3 - M1/R^3 + 3(M1.R)R/R^5]."""
    M = np.zeros(oracle.ncoef(1))
    M[0] = 2.3
    M1 = np.array([0.11, -0.07, 0.05])
    M[1:4] = M1
    R = np.array([1.3, -0.4, 2.2])
    L = oracle.m2l(1, M, R)
    r = np.linalg.norm(R)
    phi = -(M[0] / r + M1 @ R / r ** 3)
    grad = M[0] * R / r ** 3 - M1 / r ** 3 + 3 * (M1 @ R) * R / r ** 5
    assert abs(L[0] - phi) < 1e-15 * abs(phi)
    # at p = 1 the gradient keeps only the monopole (|n| + |k| <= 1)
    np.testing.assert_allclose(L[1:4], M[0] * R / r ** 3, rtol=1e-15)
    L2 = oracle.m2l(2, np.concatenate([M, np.zeros(6)]), R)
    np.testing.assert_allclose(L2[1:4], grad, rtol=1e-14)


def test_m2l_single_pair_converges_to_direct_sum():
    """Well-separated clusters: error vs direct sum falls geometrically with p."""
    rng = np.random.default_rng(7)
    src = rng.random((50, 3)) * 0.2
    msrc = rng.uniform(0.5, 1.0, 50)
    rcv = rng.random((20, 3)) * 0.2 + np.array([1.0, 0.3, -0.2])
    cB, cA = src.mean(axis=0), rcv.mean(axis=0)
    pos = np.vstack([src, rcv])
    mass = np.concatenate([msrc, np.zeros(20)])
    acc_ref, pot_ref = oracle.direct_sum(pos, mass, targets=np.arange(50, 70))
    errs = []
    for p in range(0, 9):
        L = oracle.m2l(p, oracle.p2m(p, src, msrc, cB), cA - cB)
        e = 0.0
        for i in range(20):
            phi, a = oracle.l2p(p, L, rcv[i] - cA)
            e = max(e, abs(phi - pot_ref[50 + i]) / abs(pot_ref[50 + i]))
        errs.append(e)
    errs = np.array(errs)
    assert np.all(errs[1:] < errs[:-1])
    assert errs[8] < 1e-6 * errs[0]


def test_l2l_is_exact_reexpansion():
    """Evaluating the parent's series at x equals evaluating the shifted series."""
    p = 6
    rng = np.random.default_rng(9)
    Lp = rng.normal(size=oracle.ncoef(p))
    e = np.array([0.12, -0.05, 0.08])
    Lc = oracle.l2l(p, Lp, e)
    for _ in range(10):
        dx = rng.normal(size=3) * 0.1
        pa, aa = oracle.l2p(p, Lp, e + dx)
        pb, ab = oracle.l2p(p, Lc, dx)
        assert abs(pa - pb) < 1e-13 * (abs(pa) + 1)
        np.testing.assert_allclose(aa, ab, rtol=1e-12, atol=1e-13)


def test_l2p_acceleration_is_minus_gradient():
    """a = -grad of the evaluated potential (central differences of the polynomial)."""
    p = 5
    rng = np.random.default_rng(2)
    L = rng.normal(size=oracle.ncoef(p))
    dx = np.array([0.03, -0.02, 0.05])
    _, a = oracle.l2p(p, L, dx)
    h = 1e-5
    g = np.zeros(3)
    for k in range(3):
        e = np.zeros(3)
        e[k] = h
        g[k] = (oracle.l2p(p, L, dx + e)[0] - oracle.l2p(p, L, dx - e)[0]) / (2 * h)
    np.testing.assert_allclose(a, -g, rtol=1e-7, atol=1e-8)


def test_l2p_taylor_coefficients():
    """L2P of a unit coefficient L_k reproduces dx^k / k!."""
    p = 4
    mi = oracle.multi_indices(p)
    dx = np.array([0.3, 0.2, -0.1])
    for i, k in enumerate(mi):
        L = np.zeros(len(mi))
        L[i] = 1.0
        phi, _ = oracle.l2p(p, L, dx)
        assert abs(phi - mono(dx, k)) < 1e-16
