"""GPU kick-drift-kick (Jaxion post, "Implementation": half kick, drift, half
kick) against the oracle's step, plus the fp64 reversibility check."""
import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W

pytestmark = pytest.mark.gpu


def test_one_step_matches_oracle_fp64():
    import torch

    from body_forces_morton_b300 import native

    w = W.KDK_REVERSIBILITY
    g = W.generate(W.WORKLOADS[1], n=4000, dtype="f64")
    vel0 = np.random.default_rng(3).normal(0.0, w.sigma_v, (4000, 3))
    pos, vel, mass = g["pos"].copy(), vel0.copy(), g["mass"]
    acc = oracle.fmm(pos, mass, w.p, w.theta, w.leaf).acc.copy()
    oracle.kdk_step(pos, vel, mass, acc, 1e-3, w.p, w.theta, w.leaf)
    tp = torch.from_numpy(g["pos"]).cuda()
    tv = torch.from_numpy(vel0).cuda()
    tm = torch.from_numpy(mass).cuda()
    with native.Plan(4000, w.p, w.theta, w.leaf, "f64") as pl:
        pl.kdk_step(tp, tv, tm, 1e-3, stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
    np.testing.assert_allclose(tp.cpu().numpy(), pos, rtol=0, atol=1e-15)
    np.testing.assert_allclose(tv.cpu().numpy(), vel, rtol=0, atol=1e-12 * np.abs(vel).max())


def test_cached_acceleration_matches_fresh_step():
    """Two steps with the cache equal two steps with a reset in between."""
    import torch

    from body_forces_morton_b300 import native

    g = W.generate(W.WORKLOADS[4], n=30000, dtype="f32")
    vel0 = np.random.default_rng(4).normal(0.0, 0.1, (30000, 3)).astype(np.float32)
    outs = []
    for reset in (False, True):
        tp = torch.from_numpy(g["pos"]).cuda()
        tv = torch.from_numpy(vel0).cuda()
        tm = torch.from_numpy(g["mass"]).cuda()
        with native.Plan(30000, 3, 0.6, 64, "f32") as pl:
            pl.kdk_step(tp, tv, tm, 1e-3)
            if reset:
                pl.kdk_reset()
            pl.kdk_step(tp, tv, tm, 1e-3)
        outs.append((tp.cpu().numpy(), tv.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


def run_forward_back(n, steps, dt=1e-3):
    import torch

    from body_forces_morton_b300 import native

    w = W.KDK_REVERSIBILITY
    g = W.generate(w, n=n, dtype="f64")
    tp = torch.from_numpy(g["pos"]).cuda()
    tv = torch.from_numpy(g["vel"]).cuda()
    tm = torch.from_numpy(g["mass"]).cuda()
    x0, v0 = g["pos"].copy(), g["vel"].copy()
    m = g["mass"]
    with native.Plan(n, w.p, w.theta, w.leaf, "f64") as pl:
        p_start = (m[:, None] * v0).sum(axis=0)
        for _ in range(steps):
            pl.kdk_step(tp, tv, tm, dt)
        x_mid = tp.cpu().numpy()
        p_mid = (m[:, None] * tv.cpu().numpy()).sum(axis=0)
        for _ in range(steps):
            pl.kdk_step(tp, tv, tm, -dt)
    x1, v1 = tp.cpu().numpy(), tv.cpu().numpy()
    side = (x0.max(axis=0) - x0.min(axis=0)).max()
    dx = np.linalg.norm(x1 - x0, axis=1) / side
    scale = np.sum(m * np.linalg.norm(v0, axis=1))
    return dx, x_mid, x0, np.linalg.norm(p_mid - p_start) / scale


# Momentum change over the 20 forward steps relative to sum_i m_i |v_i|: the
# force conserves momentum to rounding, so the kicks do too. Measured on a B300:
# plain step 3.4e-15, lattice step 4.5e-14 (each kick rounds every increment to
# the 2^-40 lattice). Gates about 10x above.
MOMENTUM_GATE_PLAIN = 5e-14
MOMENTUM_GATE_LATTICE = 5e-13


def test_plain_float_reversibility_report_fp64():
    """Config-5 companion with the plain float step: N = 2^18 fp64, 20 steps
    forward then 20 back. This step does NOT meet the 1e-9 bar for every
    particle: unsoftened close encounters (omega dt > 1) amplify rounding when
    run backwards, so a few particles return with errors near 1e-2 while the
    bulk returns to ~1e-11. The max and p99.9 are printed (and reported by the
    benchmark); the gate here is the median and momentum. The
    1e-9 bar for every particle is met, exactly, by the lattice step below."""
    dx, x_mid, x0, dp = run_forward_back(1 << 18, 20)
    moved = np.max(np.abs(x_mid - x0))
    print(f"plain reversibility: max {dx.max():.3e} p99.9 {np.percentile(dx, 99.9):.3e} "
          f"p99 {np.percentile(dx, 99):.3e} median {np.median(dx):.3e}; moved {moved:.3e}; |dP|/sum m|v| {dp:.3e}")
    assert moved > 1e-6
    assert np.median(dx) < 1e-9
    assert dp <= MOMENTUM_GATE_PLAIN


def snap(a, e):
    return np.rint(a * 2.0 ** (-e)) * 2.0 ** e


def test_lattice_reversibility_fp64_2p18():
    """Config-5 companion with the integer-lattice step (JZ-FMM page, "Why
    reversibility matters"): 20 steps dt = 1e-3 forward, 20 back, N = 2^18 fp64;
    the initial positions come back bit for bit (relative error 0 <= 1e-9)."""
    import torch

    from body_forces_morton_b300 import native

    w = W.KDK_REVERSIBILITY
    n = 1 << 18
    g = W.generate(w, n=n, dtype="f64")
    x0, v0 = snap(g["pos"], -40), snap(g["vel"], -40)
    tp = torch.from_numpy(g["pos"].copy()).cuda()
    tv = torch.from_numpy(g["vel"].copy()).cuda()
    tm = torch.from_numpy(g["mass"]).cuda()
    m = g["mass"]
    with native.Plan(n, w.p, w.theta, w.leaf, "f64") as pl:
        for _ in range(20):
            pl.kdk_step_lattice(tp, tv, tm, 1e-3)
        x_mid = tp.cpu().numpy()
        dp = np.linalg.norm((m[:, None] * (tv.cpu().numpy() - v0)).sum(axis=0)) / np.sum(m * np.linalg.norm(v0, axis=1))
        for _ in range(20):
            pl.kdk_step_lattice(tp, tv, tm, -1e-3)
    x1, v1 = tp.cpu().numpy(), tv.cpu().numpy()
    side = (x0.max(axis=0) - x0.min(axis=0)).max()
    err = np.max(np.linalg.norm(x1 - x0, axis=1)) / side
    print(f"lattice reversibility: max {err:.3e}; moved {np.max(np.abs(x_mid - x0)):.3e}; |dP|/sum m|v| {dp:.3e}")
    assert np.max(np.abs(x_mid - x0)) > 1e-6
    assert err <= 1e-9
    assert dp <= MOMENTUM_GATE_LATTICE
    assert np.array_equal(x1, x0) and np.array_equal(v1, v0)


def test_lattice_step_matches_oracle():
    """One lattice step against the oracle's: increments agree to one lattice unit
    (the rounded increment can flip where the fp64 forces differ by rounding)."""
    import torch

    from body_forces_morton_b300 import native

    w = W.KDK_REVERSIBILITY
    g = W.generate(W.WORKLOADS[1], n=4000, dtype="f64")
    pos = snap(g["pos"], -40)
    vel = snap(np.random.default_rng(3).normal(0.0, w.sigma_v, (4000, 3)), -40)
    mass = g["mass"]
    tp, tv, tm = (torch.from_numpy(a.copy()).cuda() for a in (pos, vel, mass))
    acc = oracle.fmm(pos, mass, w.p, w.theta, w.leaf).acc.copy()
    oracle.kdk_lattice_step(pos, vel, mass, acc, 1e-3, -40, -40, w.p, w.theta, w.leaf)
    with native.Plan(4000, w.p, w.theta, w.leaf, "f64") as pl:
        pl.kdk_step_lattice(tp, tv, tm, 1e-3)
    assert np.max(np.abs(tp.cpu().numpy() - pos)) <= 2 * 2.0 ** -40
    assert np.max(np.abs(tv.cpu().numpy() - vel)) <= 2 * 2.0 ** -40
