"""The rotation-based M2L (fmm_plan_set_m2l_rotation; jaccpot issue 152,
item 1: rotate each multipole so that the separation lies on z, translate
along z, rotate back, the rotations built on chip) against the oracle. It keeps
the same total-degree truncation as the Cartesian M2L, so the M2L locals, the
complete locals and the accelerations must meet the same gates as the default
operator: per-node local polynomials within 1e-11 (fp64) / 5e-4 (fp32), per
particle accelerations within 1e-10 / 1e-4, tree and lists bit-exact."""
import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W
from gpu_helpers import ALL_STRUCT, TOL_ACC, accel_error, assert_structure_equal, gpu_eval, local_error, pot_error

pytestmark = pytest.mark.gpu

COEFF_TOL = {"f64": 1e-11, "f32": 5e-4}


def rotation_parity(pos, mass, p, theta, leaf):
    dt = "f32" if pos.dtype == np.float32 else "f64"
    acc, pot, ex, st = gpu_eval(pos, mass, p, theta, leaf, exports=ALL_STRUCT + ("local_m2l", "local"),
                                m2l_rotation=True)
    r = oracle.fmm(pos, mass, p, theta, leaf)
    assert_structure_equal(ex, r)
    nn, nc = len(r.first), oracle.ncoef(p)
    el2 = local_error(ex["local_m2l"].reshape(nn, nc).astype(np.float64), r.Lm2l, r, p)
    el = local_error(ex["local"].reshape(nn, nc).astype(np.float64), r.L, r, p)
    if len(mass) == 1:
        assert np.all(acc == 0) and np.all(pot == 0)
        return
    e = accel_error(acc.astype(np.float64), r.acc)
    ep = pot_error(pot.astype(np.float64), r.pot)
    print(f"rotation M2L N={len(mass)} {dt} p={p}: m2l locals {el2:.2e}, locals {el:.2e}, acc {e.max():.2e}, "
          f"pot {ep.max():.2e}")
    assert el2 < COEFF_TOL[dt] and el < COEFF_TOL[dt]
    assert e.max() <= TOL_ACC[dt] and ep.max() <= TOL_ACC[dt]


@pytest.mark.parametrize("cfg", [1, 2])
def test_configs_rotation_fp64(cfg):
    w = W.WORKLOADS[cfg]
    g = W.generate(w)
    rotation_parity(g["pos"], g["mass"], w.p, w.theta, w.leaf)


@pytest.mark.parametrize("p", range(9))
def test_every_order_rotation_fp64(p):
    g = W.generate(W.WORKLOADS[2], n=5000)
    rotation_parity(g["pos"], g["mass"], p, 0.6, 16)


@pytest.mark.parametrize("p", [2, 4, 6, 8])
def test_orders_rotation_fp32_clustered(p):
    w = W.WORKLOADS[4]
    g = W.generate(w, n=65536)
    rotation_parity(g["pos"], g["mass"], p, w.theta, w.leaf)


@pytest.mark.parametrize("dt", ["f32", "f64"])
@pytest.mark.parametrize("n,leaf", [(1, 1), (2, 1), (33, 1), (4097, 8)])
def test_ragged_rotation(dt, n, leaf):
    g = W.generate(W.WORKLOADS[1], n=n, dtype=dt)
    rotation_parity(g["pos"], g["mass"], 4, 0.7, leaf)


def test_axis_aligned_separations():
    """Points on a lattice: many M2L separations lie exactly on a coordinate axis, including +-z, where
    the azimuth of the separation is undefined."""
    ax = np.arange(8, dtype=np.float64) / 8.0
    pos = np.stack(np.meshgrid(ax, ax, ax, indexing="ij"), axis=-1).reshape(-1, 3).copy()
    mass = np.full(len(pos), 1.0 / len(pos))
    rotation_parity(pos, mass, 5, 0.5, 1)
