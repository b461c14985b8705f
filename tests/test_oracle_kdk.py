"""Pins of the oracle's kick-drift-kick steps and of the walk's split rule by
results the mathematics fixes, not by properties any time-symmetric update or
any split choice would pass.

* Two equal masses on a circular orbit (Jaxion post, "Implementation": half
  kick, full drift, half kick). With G = 1, masses m = 1/2 at separation
  d = 1, each body moves on a circle of radius 1/2 at speed
  v = sqrt(G m / (2 d)) = 1/2, angular frequency 1. Two particles in one leaf
  interact by the exact direct sum, so the only error is the integrator's:
  leapfrog is second order, so the position error after a quarter period is
  small and falls by about 4 when dt halves. A full kick in place of a half
  kick, a half drift, or a drift before the first kick breaks one of the two.
  The integer-lattice step (JZ-FMM page, "Why reversibility matters") must
  behave the same when its lattice spacing is far below the per-step motion.
* The walk's split rule (symmetric dual-tree traversal: split the node with
  the larger |l|, the lower index on a tie, never a leaf). Two crafted
  four-particle inputs make the lists depend on which node is split: only the
  stated rule gives the lists asserted below.
"""
import numpy as np
import pytest

import oracle

CENTRE = np.array([0.5, 0.5, 0.5])


def orbit_state(t):
    """Positions and velocities of the two bodies at time t (omega = 1)."""
    c, s = np.cos(t), np.sin(t)
    x1 = CENTRE + 0.5 * np.array([c, s, 0.0])
    v1 = 0.5 * np.array([-s, c, 0.0])
    pos = np.stack([x1, 2 * CENTRE - x1])
    vel = np.stack([v1, -v1])
    return np.ascontiguousarray(pos), np.ascontiguousarray(vel)


def integrate(steps, lattice_exp=None):
    t_end = 0.5 * np.pi
    dt = t_end / steps
    pos, vel = orbit_state(0.0)
    mass = np.array([0.5, 0.5])
    if lattice_exp is not None:
        q = 2.0 ** lattice_exp
        pos, vel = np.rint(pos / q) * q, np.rint(vel / q) * q
    acc = oracle.fmm(pos, mass, 4, 0.7, 2).acc.copy()
    for _ in range(steps):
        if lattice_exp is None:
            oracle.kdk_step(pos, vel, mass, acc, dt, 4, 0.7, 2)
        else:
            oracle.kdk_lattice_step(pos, vel, mass, acc, dt, lattice_exp, lattice_exp, 4, 0.7, 2)
    want_pos, want_vel = orbit_state(t_end)
    return np.abs(pos - want_pos).max(), np.abs(vel - want_vel).max()


def test_two_body_force_is_exact():
    """The starting acceleration is the closed form G m / d^2 toward the other body."""
    pos, _ = orbit_state(0.3)
    r = oracle.fmm(pos, np.array([0.5, 0.5]), 4, 0.7, 2)
    want = 0.5 * (pos[1] - pos[0])  # G m / d^2 times the unit vector, d = 1
    np.testing.assert_allclose(r.acc[0], want, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r.acc[1], -want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("lattice_exp", [None, -40])
def test_kdk_second_order_on_circular_orbit(lattice_exp):
    e1, ev1 = integrate(50, lattice_exp)
    e2, ev2 = integrate(100, lattice_exp)
    print(f"lattice {lattice_exp}: quarter-period position error {e1:.3e} -> {e2:.3e} (ratio {e1 / e2:.3f}); "
          f"velocity {ev1:.3e} -> {ev2:.3e}")
    # leapfrog's phase error over a quarter period at omega dt = pi/100 is ~1e-4
    assert e1 < 3e-4 and ev1 < 3e-4
    assert 3.6 < e1 / e2 < 4.4
    assert 3.6 < ev1 / ev2 < 4.4


def test_kdk_conserves_energy_and_momentum_on_orbit():
    """Leapfrog keeps the two-body energy bounded (no drift over 4 periods) and
    momentum at zero to rounding (the pair forces are equal and opposite)."""
    pos, vel = orbit_state(0.0)
    mass = np.array([0.5, 0.5])
    acc = oracle.fmm(pos, mass, 4, 0.7, 2).acc.copy()

    def energy():
        d = np.linalg.norm(pos[0] - pos[1])
        return 0.5 * np.sum(mass[:, None] * vel ** 2) - mass[0] * mass[1] / d

    e0 = energy()
    dt = 2 * np.pi / 200
    worst = 0.0
    for _ in range(800):
        oracle.kdk_step(pos, vel, mass, acc, dt, 4, 0.7, 2)
        worst = max(worst, abs(energy() - e0))
    assert worst < 1e-3 * abs(e0)
    assert np.abs((mass[:, None] * vel).sum(axis=0)).max() < 1e-15


def line_particles(xs):
    pos = np.zeros((len(xs), 3))
    pos[:, 0] = xs
    pos[:, 1] = 0.25
    pos[:, 2] = 0.75
    return pos


def node_of(r, particles):
    """Index of the node holding exactly these original particles (the deepest one)."""
    want = set(particles)
    hits = [a for a in range(r.n_nodes) if set(r.perm[r.first[a]:r.first[a] + r.count[a]].tolist()) == want]
    return max(hits)


def top_node_of(r, particles):
    want = set(particles)
    hits = [a for a in range(r.n_nodes) if set(r.perm[r.first[a]:r.first[a] + r.count[a]].tolist()) == want]
    return min(hits)


def test_walk_splits_the_larger_node():
    """A = {0, 0.175} (|l| = 0.0875) and B = {0.625, 0.875} (|l| = 0.125) are
    the root's children; theta = 0.3 rejects (A, B) but accepts A against each
    particle of B. Splitting the larger node (B, the higher index) gives
    M2L(A <- b_j) both ways; splitting A would give pairs of A's particles with
    B instead."""
    pos = line_particles([0.0, 0.175, 0.625, 0.875])
    r = oracle.fmm(pos, np.full(4, 0.25), 2, 0.3, 1)
    A, B = top_node_of(r, [0, 1]), top_node_of(r, [2, 3])
    assert r.parent[A] == 0 and r.parent[B] == 0 and A < B
    b1, b2 = node_of(r, [2]), node_of(r, [3])
    # (B, B) pairs B's two particles with each other; (A, B) split at B pairs A with each of them
    assert r.m2l_list(A).tolist() == sorted([b1, b2])
    assert r.m2l_list(b1).tolist() == sorted([A, b2]) and r.m2l_list(b2).tolist() == sorted([A, b1])
    assert len(r.m2l_list(B)) == 0


def test_walk_splits_the_lower_index_on_a_tie():
    """A = {0, 0.25} and B = {0.625, 0.875} have exactly equal |l| = 0.125;
    the tie splits A (the lower index), so each particle of A pairs with B."""
    pos = line_particles([0.0, 0.25, 0.625, 0.875])
    r = oracle.fmm(pos, np.full(4, 0.25), 2, 0.3, 1)
    A, B = top_node_of(r, [0, 1]), top_node_of(r, [2, 3])
    assert A < B and np.array_equal(r.half[A], r.half[B])
    a1, a2 = node_of(r, [0]), node_of(r, [1])
    assert r.m2l_list(B).tolist() == sorted([a1, a2])
    assert r.m2l_list(a1).tolist() == sorted([B, a2]) and r.m2l_list(a2).tolist() == sorted([B, a1])
    assert len(r.m2l_list(A)) == 0
