"""fp64 plans with every stage in IEEE fp64 (fmm_plan_set_f64_ieee): the same
structure and the same parity gate (1e-10) against the fp64 oracle as the
default double-float stages, at the configurations' own sizes and on ragged
inputs, including split P2P receivers."""
import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W
from gpu_helpers import ALL_STRUCT, accel_error, assert_structure_equal, gpu_eval, pot_error

pytestmark = pytest.mark.gpu


def ieee_parity(pos, mass, p, theta, leaf, tol=1e-10):
    acc, pot, ex, st = gpu_eval(pos, mass, p, theta, leaf, exports=ALL_STRUCT, f64_ieee=True)
    r = oracle.fmm(pos, mass, p, theta, leaf)
    assert_structure_equal(ex, r)
    if len(mass) == 1:  # a lone particle feels nothing (the relative error is 0 / 0)
        assert np.all(acc == 0) and np.all(pot == 0)
        return acc, pot
    e, ep = accel_error(acc, r.acc), pot_error(pot, r.pot)
    print(f"IEEE fp64 N={len(mass)} p={p}: acc max {e.max():.2e}, pot max {ep.max():.2e}")
    assert e.max() <= tol and ep.max() <= tol
    return acc, pot


@pytest.mark.parametrize("cfg", [1, 2])
def test_configs_ieee(cfg):
    w = W.WORKLOADS[cfg]
    g = W.generate(w)
    ieee_parity(g["pos"], g["mass"], w.p, w.theta, w.leaf)


def test_config3_full_size_ieee():
    w = W.WORKLOADS[3]
    g = W.generate(w)
    ieee_parity(g["pos"], g["mass"], w.p, w.theta, w.leaf)


@pytest.mark.parametrize("p", [0, 2, 5, 8])
def test_orders_ieee(p):
    g = W.generate(W.WORKLOADS[2], n=6000)
    ieee_parity(g["pos"], g["mass"], p, 0.6, 16)


@pytest.mark.parametrize("n,leaf", [(1, 1), (2, 1), (33, 1), (4097, 8)])
def test_ragged_ieee(n, leaf):
    g = W.generate(W.WORKLOADS[1], n=n)
    ieee_parity(g["pos"], g["mass"], 4, 0.7, leaf)


def test_split_receivers_ieee_and_determinism():
    rng = np.random.default_rng(21)
    pos = np.vstack([0.5 + 0.02 * rng.standard_normal((60000, 3)), rng.random((40, 3))])
    mass = np.full(len(pos), 1.0 / len(pos))
    acc, pot, _, _ = gpu_eval(pos, mass, 4, 0.7, 64, f64_ieee=True)
    mask = np.zeros(len(pos), bool)
    mask[-40:] = True
    mask[rng.choice(60000, 500, replace=False)] = True
    r = oracle.fmm(pos, mass, 4, 0.7, 64, eval_mask=mask)
    assert accel_error(acc[mask], r.acc[mask]).max() <= 1e-10
    assert pot_error(pot[mask], r.pot[mask]).max() <= 1e-10
    a2, p2, _, _ = gpu_eval(pos, mass, 4, 0.7, 64, repeat=2, f64_ieee=True)
    assert np.array_equal(acc, a2) and np.array_equal(pot, p2)


def test_ieee_rejected_on_f32_plans():
    from body_forces_morton_b300 import native

    with pytest.raises(native.FmmError):
        native.Plan(100, 4, 0.7, 8, "f32", f64_ieee=True)
