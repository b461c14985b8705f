"""Pins of the oracle's whole FMM evaluation against the direct sum.

* brute force on 2..64 particles over leaf sizes, orders and opening angles,
  within a rigorous per-particle bound: for an accepted pair the truncated
  series is the degree-p Taylor polynomial of 1/|R + u| with
  |u| <= |l_A| + |l_B| = rho R, whose remainder is at most
  rho^{p+1} / ((1 - rho) R) for the potential and
  sum_{n > p} n rho^{n-1} / R^2 for the gradient (Legendre bounds);
* theta -> 0 accepts nothing, so the FMM is the direct sum to rounding;
* point-mass and shell fields through the full FMM, error shrinking with p;
* error against the direct sum falls as p rises and as theta falls;
* Newton's third law for the near field;
* fp64 kick-drift-kick reversibility (Jaxion post, `_update` loop).
"""
import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W


def remainder_bounds(r, pos, mass):
    """Per-particle bound on |dPhi| and |da| from the accepted M2L pairs."""
    n = r.n
    nn = r.n_nodes
    node_pot = np.zeros(nn)
    node_acc = np.zeros(nn)
    lnorm = np.linalg.norm(r.half, axis=1)
    m_node = np.array([mass[r.perm[r.first[a]:r.first[a] + r.count[a]]].sum() for a in range(nn)])
    p = r.p
    for a in range(nn):
        for b in r.m2l_src[r.m2l_off[a]:r.m2l_off[a + 1]]:
            R = np.linalg.norm(r.centre[a] - r.centre[b])
            rho = (lnorm[a] + lnorm[b]) / R
            assert rho < 1.0
            node_pot[a] += m_node[b] * rho ** (p + 1) / ((1 - rho) * R)
            ks = np.arange(p + 1, p + 400)
            node_acc[a] += m_node[b] * np.sum(ks * rho ** (ks - 1)) / R ** 2
    # accumulate down the tree (parents precede children)
    for a in range(1, nn):
        node_pot[a] += node_pot[r.parent[a]]
        node_acc[a] += node_acc[r.parent[a]]
    bp = np.zeros(n)
    ba = np.zeros(n)
    for a in range(nn):
        if r.nchild[a] == 0:
            idx = r.perm[r.first[a]:r.first[a] + r.count[a]]
            bp[idx] = node_pot[a]
            ba[idx] = node_acc[a]
    return bp, ba


@pytest.mark.parametrize("n", [2, 3, 9, 17, 40, 64])
@pytest.mark.parametrize("leaf", [1, 2, 4])
@pytest.mark.parametrize("theta", [0.3, 0.5, 0.7])
def test_brute_force_small(n, leaf, theta):
    for dist in (1, 2):
        g = W.generate(W.WORKLOADS[dist], n=n)
        acc_d, pot_d = oracle.direct_sum(g["pos"], g["mass"])
        for p in range(2, 7):
            r = oracle.fmm(g["pos"], g["mass"], p, theta, leaf)
            bp, ba = remainder_bounds(r, g["pos"], g["mass"])
            scale_p = np.abs(pot_d) + 1e-300
            scale_a = np.linalg.norm(acc_d, axis=1) + 1e-300
            assert np.all(np.abs(r.pot - pot_d) <= bp * (1 + 1e-9) + 1e-13 * scale_p)
            assert np.all(np.linalg.norm(r.acc - acc_d, axis=1) <= ba * (1 + 1e-9) + 1e-12 * scale_a)


def test_tiny_theta_is_direct_sum():
    g = W.generate(W.WORKLOADS[2], n=3000)
    acc_d, pot_d = oracle.direct_sum(g["pos"], g["mass"])
    r = oracle.fmm(g["pos"], g["mass"], 4, 1e-6, 16)
    np.testing.assert_allclose(r.pot, pot_d, rtol=1e-12)
    e = np.linalg.norm(r.acc - acc_d, axis=1) / np.linalg.norm(acc_d, axis=1)
    assert e.max() < 1e-10


def test_bound_holds_on_plummer():
    g = W.generate(W.WORKLOADS[2], n=3000)
    acc_d, pot_d = oracle.direct_sum(g["pos"], g["mass"])
    for p, theta in ((3, 0.5), (4, 0.7), (6, 0.4)):
        r = oracle.fmm(g["pos"], g["mass"], p, theta, 16)
        bp, ba = remainder_bounds(r, g["pos"], g["mass"])
        assert np.all(np.abs(r.pot - pot_d) <= bp + 1e-13 * np.abs(pot_d))
        assert np.all(np.linalg.norm(r.acc - acc_d, axis=1) <= ba + 1e-12 * np.linalg.norm(acc_d, axis=1))


def floored_err(acc, ref):
    na = np.linalg.norm(ref, axis=1)
    return np.linalg.norm(acc - ref, axis=1) / np.maximum(na, 1e-3 * np.median(na))


def test_error_falls_with_p_and_theta():
    """Config-3 style sweep at reduced N: rms error decreases along p and theta."""
    g = W.generate(W.WORKLOADS[3], n=6000)
    acc_d, _ = oracle.direct_sum(g["pos"], g["mass"])
    rms = {}
    for theta in (0.4, 0.5, 0.7):
        for p in (2, 3, 4, 5, 6):
            r = oracle.fmm(g["pos"], g["mass"], p, theta, 32)
            e = floored_err(r.acc, acc_d)
            rms[p, theta] = np.sqrt(np.mean(e ** 2))
    for theta in (0.4, 0.5, 0.7):
        assert all(rms[p + 1, theta] < rms[p, theta] for p in (2, 3, 4, 5))
    for p in (2, 3, 4, 5, 6):
        assert rms[p, 0.4] < rms[p, 0.5] < rms[p, 0.7]


def test_point_mass_and_shell_through_fmm():
    """Zero-mass probes far from / inside a massive shell, through M2L."""
    k = 4000
    i = np.arange(k) + 0.5
    z = 1 - 2 * i / k
    rr = np.sqrt(1 - z * z)
    ph = i * np.pi * (3 - np.sqrt(5))
    shell = np.stack([rr * np.cos(ph), rr * np.sin(ph), z], axis=1)
    rng = np.random.default_rng(8)
    probes_out = rng.normal(size=(300, 3))
    probes_out = 3.0 * probes_out / np.linalg.norm(probes_out, axis=1, keepdims=True)
    probes_in = rng.random((300, 3)) * 0.4 - 0.2
    pos = np.vstack([shell, probes_out, probes_in])
    mass = np.concatenate([np.full(k, 1.0 / k), np.zeros(600)])
    acc_d, pot_d = oracle.direct_sum(pos, mass)
    errs = []
    for p in (2, 4, 6):
        r = oracle.fmm(pos, mass, p, 0.5, 2)
        assert r.n_m2l_pairs > 0
        e = np.abs(r.pot[k:] - pot_d[k:]) / np.abs(pot_d[k:])
        errs.append(e.max())
        # shell theorem through the FMM: point-mass field outside, -1/R_s inside
        ro = np.linalg.norm(probes_out, axis=1)
        assert np.max(np.abs(r.pot[k:k + 300] * ro + 1.0)) < 5e-3
        assert np.max(np.abs(r.pot[k + 300:] + 1.0)) < 5e-3
    assert errs[0] > errs[1] > errs[2]


def test_near_field_conserves_momentum():
    """P2P alone (theta -> 0) obeys Newton's third law to rounding."""
    g = W.generate(W.WORKLOADS[4], n=4000, dtype="f64")
    r = oracle.fmm(g["pos"], g["mass"], 4, 1e-6, 64)
    m = g["mass"]
    ptot = np.sum(m[:, None] * r.acc, axis=0)
    assert np.linalg.norm(ptot) <= 1e-12 * np.sum(m * np.linalg.norm(r.acc, axis=1))


@pytest.mark.parametrize("wi,n", [(1, 4096), (2, 6000), (4, 6000)])
def test_full_fmm_conserves_momentum(wi, n):
    """With the total-degree truncation |n| + |k| <= p, the far-field forces of
    an accepted pair are equal and opposite: summed over A's particles, L2P of
    A's local gives -sum_k M_k(A) L_{k+e}(A), and D^m(-R) = (-1)^|m| D^m(R)
    turns B's sum into its negative (the index set is symmetric in n and k).
    L2L, M2M and P2M are exact polynomial identities, P2P pairs are symmetric,
    so the whole evaluation conserves momentum to rounding. A dropped parity
    factor, a transposed M2L operand, a wrong gradient index in L2P or a
    truncation that is not symmetric breaks it."""
    g = W.generate(W.WORKLOADS[wi], n=n, dtype="f64")
    m = g["mass"]
    for p, theta in ((2, 0.7), (4, 0.5), (5, 0.7)):
        r = oracle.fmm(g["pos"], m, p, theta, 16)
        ptot = np.sum(m[:, None] * r.acc, axis=0)
        assert np.linalg.norm(ptot) <= 1e-14 * np.sum(m * np.linalg.norm(r.acc, axis=1)), (p, theta)


def test_eval_mask_matches_full():
    g = W.generate(W.WORKLOADS[2], n=5000)
    full = oracle.fmm(g["pos"], g["mass"], 4, 0.7, 32)
    mask = np.zeros(5000, bool)
    mask[::97] = True
    part = oracle.fmm(g["pos"], g["mass"], 4, 0.7, 32, eval_mask=mask)
    np.testing.assert_array_equal(part.acc[mask], full.acc[mask])
    np.testing.assert_array_equal(part.pot[mask], full.pot[mask])
    assert np.all(np.isnan(part.pot[~mask]))


def test_f32_inputs_share_tree_with_widened_copy():
    """The fp32 oracle computes expansions in fp64 from the exactly widened inputs."""
    g = W.generate(W.WORKLOADS[4], n=6000, dtype="f32")
    r32 = oracle.fmm(g["pos"], g["mass"], 4, 0.7, 64)
    acc_d, _ = oracle.direct_sum(g["pos"].astype(np.float64), g["mass"].astype(np.float64))
    assert np.median(floored_err(r32.acc, acc_d)) < 1e-2


def test_kdk_reversible_fp64():
    """20 steps forward then 20 with -dt return to the start (fp64).

    A small uniform cube with the workload's velocity dispersion: at a few
    thousand particles the clustered set has close encounters (no softening)
    whose chaos amplifies rounding beyond the 1e-9 gate within 40 steps."""
    w = W.KDK_REVERSIBILITY
    g = W.generate(W.WORKLOADS[1], n=3000, dtype="f64")
    pos, mass = g["pos"].copy(), g["mass"]
    vel = np.random.default_rng(5).normal(0.0, w.sigma_v, (3000, 3))
    r0 = oracle.fmm(pos, mass, w.p, w.theta, w.leaf)
    acc = r0.acc.copy()
    x0, v0 = pos.copy(), vel.copy()
    for _ in range(20):
        oracle.kdk_step(pos, vel, mass, acc, 1e-3, w.p, w.theta, w.leaf)
    assert np.max(np.abs(pos - x0)) > 1e-5
    for _ in range(20):
        oracle.kdk_step(pos, vel, mass, acc, -1e-3, w.p, w.theta, w.leaf)
    side = (x0.max(axis=0) - x0.min(axis=0)).max()
    assert np.max(np.linalg.norm(pos - x0, axis=1)) / side < 1e-9
    assert np.max(np.linalg.norm(vel - v0, axis=1)) / np.max(np.linalg.norm(v0, axis=1)) < 1e-9


def snap(a, e):
    return np.rint(a * 2.0 ** (-e)) * 2.0 ** e


def test_lattice_kdk_is_exactly_reversible():
    """Integer-lattice KDK (JZ-FMM page, "Why reversibility matters"): 10 steps
    forward and 10 back return the lattice state bit for bit, here on the
    clustered recipe whose close encounters defeat the plain float step."""
    w = W.KDK_REVERSIBILITY
    g = W.generate(w, n=3000, dtype="f64")
    pos = snap(g["pos"], -40)
    vel = snap(g["vel"], -40)
    mass = g["mass"]
    x0, v0 = pos.copy(), vel.copy()
    acc = oracle.fmm(pos, mass, w.p, w.theta, w.leaf).acc.copy()
    for _ in range(10):
        oracle.kdk_lattice_step(pos, vel, mass, acc, 1e-3, -40, -40, w.p, w.theta, w.leaf)
    assert np.max(np.abs(pos - x0)) > 1e-6
    for _ in range(10):
        oracle.kdk_lattice_step(pos, vel, mass, acc, -1e-3, -40, -40, w.p, w.theta, w.leaf)
    assert np.array_equal(pos, x0) and np.array_equal(vel, v0)
