"""Pins of the oracle's O(N^2) direct sum against closed forms and invariants.

The direct sum is the definition the FMM approximates (JZ-FMM page, "From
particle pairs to node pairs": Phi(x_i) = -G sum_{j != i} m_j / |x_i - x_j|,
self-interaction omitted; a = -grad Phi). G = 1.
"""
import math

import numpy as np
import pytest

import oracle


def fibonacci_sphere(k, radius):
    i = np.arange(k) + 0.5
    z = 1.0 - 2.0 * i / k
    rho = np.sqrt(1.0 - z * z)
    phi = i * math.pi * (3.0 - math.sqrt(5.0))
    return radius * np.stack([rho * np.cos(phi), rho * np.sin(phi), z], axis=1)


def test_point_mass_closed_form():
    """Zero-mass probes around one mass M: Phi = -M/r, a = -M r_hat / r^2."""
    rng = np.random.default_rng(11)
    M = 2.5
    centre = np.array([0.3, -0.2, 0.7])
    probes = centre + rng.normal(size=(50, 3)) * rng.uniform(0.1, 5.0, size=(50, 1))
    pos = np.vstack([centre, probes])
    mass = np.concatenate([[M], np.zeros(50)])
    acc, pot = oracle.direct_sum(pos, mass)
    d = probes - centre
    r = np.linalg.norm(d, axis=1)
    np.testing.assert_allclose(pot[1:], -M / r, rtol=1e-14)
    np.testing.assert_allclose(acc[1:], -M * d / r[:, None] ** 3, rtol=1e-13, atol=0)
    # the source feels nothing from massless probes, and no self force
    assert pot[0] == 0.0 and np.all(acc[0] == 0.0)


@pytest.mark.parametrize("k", [1000, 4000, 16000])
def test_uniform_shell(k):
    """Shell theorem: outside = point mass; inside = constant -M/R_s, zero force."""
    M, Rs = 1.0, 1.0
    shell = fibonacci_sphere(k, Rs)
    rng = np.random.default_rng(5)
    dirs = rng.normal(size=(20, 3))
    dirs /= np.linalg.norm(dirs, axis=1, keepdims=True)
    outside = dirs[:10] * rng.uniform(2.0, 4.0, size=(10, 1))
    inside = dirs[10:] * rng.uniform(0.0, 0.4, size=(10, 1))
    pos = np.vstack([shell, outside, inside])
    mass = np.concatenate([np.full(k, M / k), np.zeros(20)])
    tgt = np.arange(k, k + 20)
    acc, pot = oracle.direct_sum(pos, mass, targets=tgt)
    ro = np.linalg.norm(outside, axis=1)
    err_out_pot = np.max(np.abs(pot[k:k + 10] + M / ro) * ro / M)
    err_out_acc = np.max(np.linalg.norm(acc[k:k + 10] + M * outside / ro[:, None] ** 3, axis=1) * ro ** 2 / M)
    err_in_pot = np.max(np.abs(pot[k + 10:] + M / Rs))
    err_in_acc = np.max(np.linalg.norm(acc[k + 10:], axis=1))
    # discretisation error of a K-point Fibonacci shell; calibrated at K = 1e4 with margin
    tol = 2e-3 * (10000.0 / k)
    assert err_out_pot < tol and err_out_acc < tol
    assert err_in_pot < tol and err_in_acc < tol


def test_shell_error_shrinks_with_k():
    errs = []
    for k in (500, 2000, 8000):
        shell = fibonacci_sphere(k, 1.0)
        probe = np.array([[0.1, 0.2, -0.15]])
        pos = np.vstack([shell, probe])
        mass = np.concatenate([np.full(k, 1.0 / k), [0.0]])
        acc, pot = oracle.direct_sum(pos, mass, targets=[k])
        errs.append(abs(pot[k] + 1.0) + np.linalg.norm(acc[k]))
    assert errs[0] > errs[1] > errs[2]


def test_energy_pair_symmetry():
    """1/2 sum_i m_i Phi_i equals -sum_{i<j} m_i m_j / r_ij (pair enumeration)."""
    rng = np.random.default_rng(3)
    n = 300
    pos = rng.random((n, 3))
    mass = rng.uniform(0.5, 2.0, n)
    _, pot = oracle.direct_sum(pos, mass)
    iu, ju = np.triu_indices(n, k=1)
    r = np.linalg.norm(pos[iu] - pos[ju], axis=1)
    w_pairs = -np.sum(mass[iu] * mass[ju] / r)
    assert abs(0.5 * np.sum(mass * pot) - w_pairs) <= 1e-13 * abs(w_pairs)


def test_newton_third_law():
    rng = np.random.default_rng(4)
    pos = rng.normal(size=(500, 3))
    mass = rng.uniform(0.1, 1.0, 500)
    acc, _ = oracle.direct_sum(pos, mass)
    p = np.sum(mass[:, None] * acc, axis=0)
    scale = np.sum(mass * np.linalg.norm(acc, axis=1))
    assert np.linalg.norm(p) <= 1e-13 * scale


def test_coincident_particles_skipped():
    """Zero-separation pairs (self or coincident) contribute nothing."""
    pos = np.array([[0.0, 0.0, 0.0], [0.0, 0.0, 0.0], [1.0, 0.0, 0.0]])
    mass = np.array([1.0, 2.0, 3.0])
    acc, pot = oracle.direct_sum(pos, mass)
    assert np.all(np.isfinite(acc)) and np.all(np.isfinite(pot))
    np.testing.assert_allclose(pot[0], -3.0, rtol=1e-15)
    np.testing.assert_allclose(acc[0], [3.0, 0.0, 0.0], rtol=1e-15)
    np.testing.assert_allclose(pot[2], -3.0, rtol=1e-15)
