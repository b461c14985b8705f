"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: keys, sort permutation, tree, node boxes and interaction lists
bit-exact; expansion coefficients per stage; accelerations within a per-particle
L2 relative error (floored at 1e-3 of the median) of 1e-10 in fp64 and 1e-4 in
fp32, potentials likewise.
"""
import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W
from gpu_helpers import (ALL_STRUCT, TOL_ACC, accel_error, assert_structure_equal, gpu_eval, local_error,
                         moment_error, pot_error)

pytestmark = pytest.mark.gpu

COEFF_TOL = {"f64": 1e-11, "f32": 5e-4}


def full_parity(pos, mass, p, theta, leaf, check_coeffs=True):
    dt = "f32" if pos.dtype == np.float32 else "f64"
    ex_names = ALL_STRUCT + (("multipole", "local_m2l", "local") if check_coeffs else ())
    acc, pot, ex, st = gpu_eval(pos, mass, p, theta, leaf, exports=ex_names)
    r = oracle.fmm(pos, mass, p, theta, leaf)
    assert_structure_equal(ex, r)
    nn = len(r.first)
    nc = oracle.ncoef(p)
    if check_coeffs:
        em = moment_error(ex["multipole"].reshape(nn, nc).astype(np.float64), r, p)
        el2 = local_error(ex["local_m2l"].reshape(nn, nc).astype(np.float64), r.Lm2l, r, p)
        el = local_error(ex["local"].reshape(nn, nc).astype(np.float64), r.L, r, p)
        print(f"N={len(mass)} {dt} p={p}: moments {em:.2e} m2l {el2:.2e} local {el:.2e}")
        assert em < COEFF_TOL[dt], f"P2M/M2M moments {em:.3e}"
        assert el2 < COEFF_TOL[dt], f"M2L locals {el2:.3e}"
        assert el < COEFF_TOL[dt], f"L2L locals {el:.3e}"
    e = accel_error(acc.astype(np.float64), r.acc)
    ep = pot_error(pot.astype(np.float64), r.pot)
    print(f"  acc error max {e.max():.2e} p99 {np.percentile(e, 99):.2e}; pot max {ep.max():.2e}")
    assert e.max() <= TOL_ACC[dt], f"max acc error {e.max():.3e}"
    assert ep.max() <= TOL_ACC[dt], f"max pot error {ep.max():.3e}"
    assert st["n_nodes"] == nn and st["n_m2l"] == len(r.m2l_src) and st["n_p2p"] == len(r.p2p_src)
    assert st["n_p2p_interactions"] == r.n_p2p_interactions
    return e, r, st


@pytest.mark.parametrize("cfg", [1, 2])
def test_small_configs_full_parity(cfg):
    w = W.WORKLOADS[cfg]
    g = W.generate(w)
    full_parity(g["pos"], g["mass"], w.p, w.theta, w.leaf)


def test_plummer_reduced_f64():
    w = W.WORKLOADS[3]
    g = W.generate(w, n=30000)
    full_parity(g["pos"], g["mass"], w.p, w.theta, w.leaf)


@pytest.mark.parametrize("n", [65536, 100003])
def test_clustered_f32(n):
    w = W.WORKLOADS[4]
    g = W.generate(w, n=n)
    full_parity(g["pos"], g["mass"], w.p, w.theta, w.leaf)


def test_kdk_config_params_f32():
    w = W.WORKLOADS[5]
    g = W.generate(w, n=70000)
    full_parity(g["pos"], g["mass"], w.p, w.theta, w.leaf)


@pytest.mark.parametrize("p", range(0, 9))
def test_every_order_f64(p):
    g = W.generate(W.WORKLOADS[2], n=3000)
    full_parity(g["pos"], g["mass"], p, 0.5, 16)


@pytest.mark.parametrize("p", [2, 5, 6])
def test_orders_f32(p):
    g = W.generate(W.WORKLOADS[4], n=20000)
    full_parity(g["pos"], g["mass"], p, 0.6, 32)


@pytest.mark.parametrize("n", [1, 2, 3, 33, 4095, 4097, 10007])
@pytest.mark.parametrize("dt", ["f64", "f32"])
@pytest.mark.parametrize("leaf", [1, 8])
def test_ragged_sizes(n, dt, leaf):
    g = W.generate(W.WORKLOADS[1], n=n, dtype=dt)
    if n == 1:
        acc, pot, ex, st = gpu_eval(g["pos"], g["mass"], 4, 0.7, leaf)
        assert np.all(acc == 0) and np.all(pot == 0) and st["n_nodes"] == 1
        return
    full_parity(g["pos"], g["mass"], 4, 0.7, leaf)


@pytest.mark.parametrize("theta", [0.05, 0.3, 1.0])
def test_opening_angles(theta):
    g = W.generate(W.WORKLOADS[2], n=5000)
    full_parity(g["pos"], g["mass"], 3, theta, 8)


def test_coincident_particles_and_depth_limit():
    """Coincident points: a depth-21 leaf holding more than `leaf` particles."""
    rng = np.random.default_rng(0)
    pos = np.vstack([np.full((100, 3), 0.5), rng.random((400, 3))])
    mass = np.full(500, 1.0 / 500)
    e, r, st = full_parity(pos, mass, 4, 0.7, 8)
    assert r.depth == 21 and st["depth"] == 21


@pytest.mark.parametrize("dt", ["f32", "f64"])
@pytest.mark.parametrize("leaf", [1, 2048, 4096, 4097, 9000])
def test_tree_window_and_level_builds(leaf, dt):
    """Leaves up to 4096 build every level at once (windows over the divergence levels of the sorted keys);
    larger leaves take the level-by-level build. Both give the oracle's tree bit for bit, across tile and
    chunk edges of the window build (40000 clustered keys, depth up to 21)."""
    n = 40000
    g = W.generate(W.WORKLOADS[4], n=n, dtype=dt)
    mask = np.zeros(n, bool)
    mask[::997] = True
    _, _, ex, st = gpu_eval(g["pos"], g["mass"], 2, 0.7, leaf, exports=ALL_STRUCT)
    r = oracle.fmm(g["pos"], g["mass"], 2, 0.7, leaf, eval_mask=mask)
    assert_structure_equal(ex, r)
    assert st["depth"] == r.depth


def test_tiny_theta_equals_direct_sum():
    g = W.generate(W.WORKLOADS[2], n=4000)
    acc, pot, _, _ = gpu_eval(g["pos"], g["mass"], 4, 1e-6, 16)
    acc_d, pot_d = oracle.direct_sum(g["pos"], g["mass"])
    assert accel_error(acc, acc_d).max() < 1e-12
    assert pot_error(pot, pot_d).max() < 1e-12


def test_deterministic_bitwise():
    g = W.generate(W.WORKLOADS[4], n=50000)
    a1, p1, _, _ = gpu_eval(g["pos"], g["mass"], 4, 0.7, 64)
    a2, p2, _, _ = gpu_eval(g["pos"], g["mass"], 4, 0.7, 64, repeat=3)
    assert np.array_equal(a1, a2) and np.array_equal(p1, p2)


def test_plan_reuse_and_pot_optional():
    import torch

    from body_forces_morton_b300 import native

    g1 = W.generate(W.WORKLOADS[1], n=5000)
    g2 = W.generate(W.WORKLOADS[2], n=5000)
    with native.Plan(5000, 4, 0.7, 32, "f64") as pl:
        a1, _, _, _ = gpu_eval(g1["pos"], g1["mass"], 4, 0.7, 32, plan=pl)
        a2, _, _, _ = gpu_eval(g2["pos"], g2["mass"], 4, 0.7, 32, plan=pl, want_pot=False)
        a1b, _, _, _ = gpu_eval(g1["pos"], g1["mass"], 4, 0.7, 32, plan=pl)
    assert np.array_equal(a1, a1b)
    r2 = oracle.fmm(g2["pos"], g2["mass"], 4, 0.7, 32)
    assert accel_error(a2, r2.acc).max() <= 1e-10


def test_eval_host_matches_device():
    from body_forces_morton_b300 import native

    g = W.generate(W.WORKLOADS[4], n=40000)
    acc_d, pot_d, _, _ = gpu_eval(g["pos"], g["mass"], 4, 0.7, 64)
    acc_h = np.empty_like(g["pos"])
    pot_h = np.empty_like(g["mass"])
    with native.Plan(40000, 4, 0.7, 64, "f32") as pl:
        pl.eval_host(g["pos"], g["mass"], acc_h, pot_h)
    assert np.array_equal(acc_h, acc_d) and np.array_equal(pot_h, pot_d)


def test_error_paths():
    import torch

    from body_forces_morton_b300 import native

    with pytest.raises(native.FmmError):
        native.Plan(0, 4, 0.7, 32, "f64")
    with pytest.raises(native.FmmError):
        native.Plan(10, 9, 0.7, 32, "f64")
    with pytest.raises(native.FmmError):
        native.Plan(10, 4, 1.5, 32, "f64")
    with native.Plan(100, 4, 0.7, 8, "f64") as pl:
        pos = torch.rand(100, 3, dtype=torch.float64, device="cuda")
        pos[17, 1] = float("nan")
        mass = torch.full((100,), 0.01, dtype=torch.float64, device="cuda")
        acc = torch.empty_like(pos)
        with pytest.raises(native.FmmError) as ei:
            pl.eval(pos, mass, acc)
        assert ei.value.status == 5
        with pytest.raises(native.FmmError) as ei:
            native.fmm_eval(pl.handle, pos, None, acc)
        assert ei.value.status == 1
        pos[17, 1] = 0.5
        pl.eval(pos, mass, acc)  # the plan stays usable after an error
        assert torch.isfinite(acc).all()


@pytest.mark.parametrize("scale,shift,mscale", [(1e-12, 0.0, 1.0), (1e9, 0.0, 1e-20), (1.0, 1e6, 1e25),
                                                (3e-30, 7e-29, 1e-3)])
def test_fp64_units_extreme_scales(scale, shift, mscale):
    """The fp64 near field runs in power-of-two units of the root box and the
    total mass; far from unit scales the result still matches the oracle."""
    g = W.generate(W.WORKLOADS[2], n=3000)
    full_parity(g["pos"] * scale + shift, g["mass"] * mscale, 4, 0.7, 32, check_coeffs=False)


@pytest.mark.parametrize("same_leaf", [False, True])
def test_fp64_close_pair(same_leaf):
    """Two particles 8e-15 apart (below 2^-42 of the box, where the near field
    switches to its wide-range form): across the root's midplane, so in
    different leaves, or inside one leaf."""
    rng = np.random.default_rng(3)
    pos = rng.random((600, 3))
    pos[2], pos[3] = 0.0, 1.0                     # root cube [0, 1]^3 exactly
    x0 = 0.5 if not same_leaf else 0.3
    pos[0] = [x0 - 4e-15, 0.3, 0.3]
    pos[1] = [x0 + 4e-15, 0.3, 0.3]
    mass = np.full(600, 1.0 / 600)
    e, r, _ = full_parity(pos, mass, 4, 0.7, 8, check_coeffs=False)
    leaf_of = np.empty(600, int)
    for a in np.flatnonzero(r.nchild == 0):
        leaf_of[r.perm[r.first[a]:r.first[a] + r.count[a]]] = a
    assert (leaf_of[0] == leaf_of[1]) == same_leaf


def _df_wide_pairs(r):
    """M2L pairs outside the ranges of the fp64 path's double-word units
    (level gap above 8, or |R / h_A|^2 outside [2^-30, 2^30] with
    h_A = 2^(ex - level_A), 2^(ex-1) <= the root's largest half-width < 2^ex)."""
    ex = np.frexp(r.half[0].max())[1]
    n = 0
    for a in range(r.n_nodes):
        src = r.m2l_list(a)
        if len(src) == 0:
            continue
        rs = (r.centre[a] - r.centre[src]) * 2.0 ** -(ex - int(r.level[a]))
        r2 = (rs.astype(np.float32).astype(np.float64) ** 2).sum(axis=1)
        dl = np.abs(int(r.level[a]) - r.level[src])
        n += int(((dl > 8) | (r2 < 2.0 ** -30) | (r2 > 2.0 ** 30)).sum())
    return n


def test_fp64_m2l_wide_pairs():
    """Two dense clumps 1e-9 apart on either side of the root's midplane: their
    nodes meet in M2L at a separation far below their cells' size, which the
    fp64 M2L evaluates in its fp64 pass; coefficients and accelerations must
    still match the oracle."""
    rng = np.random.default_rng(11)
    bg = rng.random((500, 3))
    bg[0], bg[1] = 0.0, 1.0
    c1 = np.array([0.5 - 5e-10, 0.3, 0.3]) + 1e-12 * rng.standard_normal((40, 3))
    c2 = np.array([0.5 + 5e-10, 0.3, 0.3]) + 1e-12 * rng.standard_normal((40, 3))
    pos = np.vstack([bg, c1, c2])
    mass = rng.uniform(0.5, 1.5, len(pos)) / len(pos)
    e, r, _ = full_parity(pos, mass, 4, 0.7, 8, check_coeffs=True)
    assert _df_wide_pairs(r) > 0


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_split_p2p_receivers(dt):
    """A dense cluster with a few particles spread over the box: the sparse
    leaves' tight boxes are large, so their P2P lists take in thousands of
    cluster leaves and their work is split into chunks that different warps
    sum in chunk order. Accelerations of the sparse particles (and a sample of
    the others) against the oracle, bitwise repeatability, and that at least
    one receiver was split (work above 2^20 interactions)."""
    rng = np.random.default_rng(21)
    pos = np.vstack([0.5 + 0.02 * rng.standard_normal((60000, 3)), rng.random((40, 3))]).astype(dt)
    mass = np.full(len(pos), 1.0 / len(pos), dtype=dt)
    acc, pot, ex, st = gpu_eval(pos, mass, 4, 0.7, 64, exports=("node_count", "p2p_off", "p2p_src"))
    cnt = ex["node_count"].astype(np.int64)
    off, src = ex["p2p_off"], ex["p2p_src"]
    work = np.array([cnt[a] * cnt[src[off[a]:off[a + 1]]].sum() for a in range(len(cnt))])
    assert work.max() > (1 << 20)
    mask = np.zeros(len(pos), bool)
    mask[-40:] = True
    mask[rng.choice(60000, 500, replace=False)] = True
    r = oracle.fmm(pos, mass, 4, 0.7, 64, eval_mask=mask)
    tol = TOL_ACC["f32" if dt == np.float32 else "f64"]
    e = accel_error(acc[mask].astype(np.float64), r.acc[mask])
    ep = pot_error(pot[mask].astype(np.float64), r.pot[mask])
    print(f"split receivers ({np.dtype(dt).name}): max work {work.max()}, acc error {e.max():.2e}, pot {ep.max():.2e}")
    assert e.max() <= tol and ep.max() <= tol
    a2, p2, _, _ = gpu_eval(pos, mass, 4, 0.7, 64, repeat=3)
    assert np.array_equal(acc, a2) and np.array_equal(pot, p2)
