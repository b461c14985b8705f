"""Pins of the oracle's FMM vector-Jacobian product (JZ-FMM page,
"Differentiating the force calculation": one contribution from the next higher
derivative of the original evaluation, one from an FMM whose sources are the
force sensitivities acting as dipoles).

The loss is l = sum_i abar_i . a_i + pbar_i phi_i with seeded random
cotangents; the VJP returns dl/dx_k and dl/dm_k.

* Operators: the dipole P2M is the directional derivative of the point-mass
  P2M; the local series' Hessian is the derivative of its gradient (central
  differences; both are polynomials, so the differences agree to ~h^2).
* theta -> 0 with one particle per leaf: every accepted pair is between two
  zero-size nodes, so the FMM is exact and its VJP must equal central
  differences of the direct sum (pinned by closed forms elsewhere).
* theta = 0.5, p = 4: the VJP is the exact derivative of the evaluation with the
  tree and the expansion centres held fixed. Moving a particle that lies strictly
  inside its leaf's box by a small step changes no centre, key or list, so
  central differences of the oracle's own evaluation must match it.
"""
import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W


def loss(pos, mass, ab, pb, p, theta, leaf):
    r = oracle.fmm(pos, mass, p, theta, leaf)
    return float(np.sum(ab * r.acc) + np.sum(pb * r.pot))


def loss_direct(pos, mass, ab, pb):
    acc, pot = oracle.direct_sum(pos, mass)
    return float(np.sum(ab * acc) + np.sum(pb * pot))


def cotangents(n, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(size=(n, 3)), rng.normal(size=n)


def test_dipole_p2m_is_directional_derivative():
    rng = np.random.default_rng(11)
    for p in (1, 2, 4, 6):
        x = rng.uniform(-0.3, 0.3, (5, 3))
        q = rng.normal(size=5)
        d = rng.normal(size=(5, 3))
        c = np.array([0.05, -0.02, 0.01])
        got = oracle.p2m_dipole(p, x, q, d, c)
        h = 1e-5
        want = oracle.p2m(p, x, q, c)
        for j in range(5):
            up = oracle.p2m(p, x[j] + h * d[j], [1.0], c)
            dn = oracle.p2m(p, x[j] - h * d[j], [1.0], c)
            want = want + (up - dn) / (2 * h)
        np.testing.assert_allclose(got, want, rtol=1e-7, atol=1e-9 * np.abs(want).max())
        # without monopoles only the dipole part remains
        np.testing.assert_allclose(oracle.p2m_dipole(p, x, None, d, c), want - oracle.p2m(p, x, q, c),
                                   rtol=1e-7, atol=1e-9 * np.abs(want).max())


def test_local_hessian_is_gradient_derivative():
    rng = np.random.default_rng(12)
    pairs = [(0, 0), (0, 1), (0, 2), (1, 1), (1, 2), (2, 2)]
    for p in (2, 3, 4, 6):
        L = rng.normal(size=oracle.ncoef(p))
        dx = rng.uniform(-0.2, 0.2, 3)
        H = oracle.l2p_hess(p, L, dx)
        h = 1e-5
        for k, (a, b) in enumerate(pairs):
            e = np.zeros(3)
            e[b] = h
            _, acc_up = oracle.l2p(p, L, dx + e)
            _, acc_dn = oracle.l2p(p, L, dx - e)
            want = -(acc_up[a] - acc_dn[a]) / (2 * h)   # acc = -grad Phi
            assert abs(H[k] - want) <= 1e-7 * max(1.0, abs(want)), (p, a, b, H[k], want)
    # p < 2: no second derivatives survive the truncation
    assert np.all(oracle.l2p_hess(1, rng.normal(size=4), dx) == 0)


@pytest.mark.parametrize("dist", [1, 2])
def test_vjp_equals_direct_sum_derivative_when_exact(dist):
    n = 40
    g = W.generate(W.WORKLOADS[dist], n=n)
    pos, mass = g["pos"], g["mass"] * np.random.default_rng(5).uniform(0.5, 1.5, n)
    ab, pb = cotangents(n, 21)
    xb, mb = oracle.fmm_vjp(pos, mass, ab, pb, p=3, theta=1e-3, leaf=1)
    h = 1e-6 * (pos.max() - pos.min())
    fd_x = np.zeros((n, 3))
    for k in range(n):
        for d in range(3):
            up, dn = pos.copy(), pos.copy()
            up[k, d] += h
            dn[k, d] -= h
            fd_x[k, d] = (loss_direct(up, mass, ab, pb) - loss_direct(dn, mass, ab, pb)) / (2 * h)
    fd_m = np.zeros(n)
    hm = 1e-6 * mass.max()
    for k in range(n):
        up, dn = mass.copy(), mass.copy()
        up[k] += hm
        dn[k] -= hm
        fd_m[k] = (loss_direct(pos, up, ab, pb) - loss_direct(pos, dn, ab, pb)) / (2 * hm)
    scale_x = np.abs(fd_x).max()
    np.testing.assert_allclose(xb, fd_x, rtol=0, atol=2e-6 * scale_x)
    np.testing.assert_allclose(mb, fd_m, rtol=0, atol=2e-6 * np.abs(fd_m).max())


def interior_particles(r, pos):
    """Original indices of particles strictly inside their leaf's box in every axis."""
    out = []
    for a in range(r.n_nodes):
        if r.nchild[a] != 0:
            continue
        for i in range(r.first[a], r.first[a] + r.count[a]):
            o = r.perm[i]
            if np.all(pos[o] > r.lo[a]) and np.all(pos[o] < r.hi[a]):
                out.append(o)
    return np.array(sorted(out))


@pytest.mark.parametrize("dtype", ["f64", "f32"])
def test_vjp_equals_fixed_structure_derivative(dtype):
    n, p, theta, leaf = 400, 4, 0.5, 16
    g = W.generate(W.WORKLOADS[2], n=n, dtype=dtype)
    pos, mass = g["pos"], g["mass"]
    ab, pb = cotangents(n, 22)
    xb, mb = oracle.fmm_vjp(pos, mass, ab, pb, p, theta, leaf)
    pos64 = pos.astype(np.float64)
    mass64 = mass.astype(np.float64)
    r0 = oracle.fmm(pos64, mass64, p, theta, leaf, tree_only=True)
    inner = interior_particles(r0, pos64)
    assert len(inner) > 50
    pick = inner[np.random.default_rng(7).choice(len(inner), 12, replace=False)]
    h = 1e-6
    for k in pick:
        for d in range(3):
            up, dn = pos64.copy(), pos64.copy()
            up[k, d] += h
            dn[k, d] -= h
            for q in (up, dn):  # the step must leave the structure untouched
                rq = oracle.fmm(q, mass64, p, theta, leaf, tree_only=True)
                assert np.array_equal(rq.perm, r0.perm) and np.array_equal(rq.m2l_src, r0.m2l_src)
                assert np.array_equal(rq.centre, r0.centre)
            fd = (loss(up, mass64, ab, pb, p, theta, leaf) - loss(dn, mass64, ab, pb, p, theta, leaf)) / (2 * h)
            assert abs(xb[k, d] - fd) <= 1e-6 * max(1.0, abs(fd)), (k, d, xb[k, d], fd)
    # masses never move a centre: every particle qualifies
    hm = 1e-6 * mass64.max()
    for k in np.random.default_rng(8).choice(n, 12, replace=False):
        up, dn = mass64.copy(), mass64.copy()
        up[k] += hm
        dn[k] -= hm
        fd = (loss(pos64, up, ab, pb, p, theta, leaf) - loss(pos64, dn, ab, pb, p, theta, leaf)) / (2 * hm)
        assert abs(mb[k] - fd) <= 1e-6 * max(1.0, abs(fd)), (k, mb[k], fd)


def test_vjp_potential_cotangent_optional_and_linear():
    n = 300
    g = W.generate(W.WORKLOADS[1], n=n)
    ab, pb = cotangents(n, 23)
    x0, m0 = oracle.fmm_vjp(g["pos"], g["mass"], ab, None, 4, 0.6, 8)
    x1, m1 = oracle.fmm_vjp(g["pos"], g["mass"], ab, np.zeros(n), 4, 0.6, 8)
    assert np.array_equal(x0, x1) and np.array_equal(m0, m1)
    x2, m2 = oracle.fmm_vjp(g["pos"], g["mass"], 2.0 * ab, 2.0 * pb, 4, 0.6, 8)
    x3, m3 = oracle.fmm_vjp(g["pos"], g["mass"], ab, pb, 4, 0.6, 8)
    np.testing.assert_allclose(x2, 2.0 * x3, rtol=1e-13, atol=1e-13 * np.abs(x3).max())
    np.testing.assert_allclose(m2, 2.0 * m3, rtol=1e-13, atol=1e-13 * np.abs(m3).max())
