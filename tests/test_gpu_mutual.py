"""The mutual evaluation (fmm_plan_set_mutual; jaccpot issue 152, "Mutual
FMM": every unordered accepted pair evaluated once for both receivers) against
the oracle and against the default evaluation.

It keeps the total-degree truncation and the lists, so it computes the same
result as the default path up to rounding: tree and lists bit-exact, M2L and
complete locals within the per-node gates (1e-11 fp64, 5e-4 fp32),
accelerations and potentials within 1e-10 / 1e-4 of the oracle. Its sums run in
a fixed order (no floating-point atomics), so repeated evaluations agree bit
for bit, and a shortened partner-share buffer regrows to the same result.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W
from gpu_helpers import ALL_STRUCT, TOL_ACC, accel_error, assert_structure_equal, gpu_eval, local_error, pot_error

pytestmark = pytest.mark.gpu

COEFF_TOL = {"f64": 1e-11, "f32": 5e-4}
# mutual against the default GPU evaluation: the same arithmetic in another order
# (and, for fp64 plans, IEEE fp64 against the double-float default), so the
# difference is rounding: fp64 ~1e-14, fp32 ~1e-6 relative per particle, floored
# as accel_error floors it; the gates leave an order of magnitude
AGREE_TOL = {"f64": 1e-12, "f32": 2e-5}
# |sum m a| / sum m |a| at the rounding level. These cases run from N = 2 to
# 65536, and at small N the per-particle rounding does not average out as it
# does over 2^20 particles: the imbalance is then of the order of the rounding
# unit itself (measured 2.0e-8 in fp32 at N = 33, 2.6e-16 in fp64), so the gates
# are two rounding units, 2 x 2^-24 and 2 x 2^-53 scaled by the 20-odd
# accumulation steps of a particle's far field (~5e-15)
MOMENTUM_GATE = {"f64": 5e-15, "f32": 1.2e-7}


def momentum_imbalance(mass, acc):
    m = np.asarray(mass, np.float64)
    a = np.asarray(acc, np.float64)
    return np.linalg.norm((m[:, None] * a).sum(axis=0)) / np.sum(m * np.linalg.norm(a, axis=1))


def mutual_parity(pos, mass, p, theta, leaf):
    dt = "f32" if pos.dtype == np.float32 else "f64"
    acc, pot, ex, st = gpu_eval(pos, mass, p, theta, leaf, exports=ALL_STRUCT + ("local_m2l", "local"), mutual=True)
    r = oracle.fmm(pos, mass, p, theta, leaf)
    assert_structure_equal(ex, r)
    if len(mass) == 1:
        assert np.all(acc == 0) and np.all(pot == 0)
        return acc, pot
    nn, nc = len(r.first), oracle.ncoef(p)
    el2 = local_error(ex["local_m2l"].reshape(nn, nc).astype(np.float64), r.Lm2l, r, p)
    el = local_error(ex["local"].reshape(nn, nc).astype(np.float64), r.L, r, p)
    e = accel_error(acc.astype(np.float64), r.acc)
    ep = pot_error(pot.astype(np.float64), r.pot)
    acc_d, pot_d, _, _ = gpu_eval(pos, mass, p, theta, leaf)
    ed = accel_error(acc.astype(np.float64), acc_d.astype(np.float64))
    dp = momentum_imbalance(mass, acc)
    print(f"mutual N={len(mass)} {dt} p={p} theta={theta} leaf={leaf}: m2l locals {el2:.2e}, locals {el:.2e}, "
          f"acc {e.max():.2e}, pot {ep.max():.2e}; against the default path {ed.max():.2e}; momentum {dp:.2e}")
    assert el2 < COEFF_TOL[dt] and el < COEFF_TOL[dt]
    assert e.max() <= TOL_ACC[dt] and ep.max() <= TOL_ACC[dt]
    assert ed.max() <= AGREE_TOL[dt]
    assert dp <= MOMENTUM_GATE[dt]
    return acc, pot


@pytest.mark.parametrize("cfg", [1, 2])
def test_configs_mutual_fp64(cfg):
    w = W.WORKLOADS[cfg]
    g = W.generate(w)
    mutual_parity(g["pos"], g["mass"], w.p, w.theta, w.leaf)


@pytest.mark.parametrize("p", range(9))
def test_every_order_mutual_fp64(p):
    g = W.generate(W.WORKLOADS[2], n=5000)
    mutual_parity(g["pos"], g["mass"], p, 0.6, 16)


@pytest.mark.parametrize("p,leaf", [(2, 64), (4, 64), (4, 100), (6, 32)])
def test_clustered_mutual_fp32(p, leaf):
    """Leaves of up to 64 and 100 particles: receivers beyond 32 take several lane blocks."""
    w = W.WORKLOADS[4]
    g = W.generate(w, n=65536)
    mutual_parity(g["pos"], g["mass"], p, w.theta, leaf)


@pytest.mark.parametrize("dt", ["f32", "f64"])
@pytest.mark.parametrize("n,leaf", [(1, 1), (2, 1), (33, 1), (4097, 8), (3000, 3)])
def test_ragged_mutual(dt, n, leaf):
    g = W.generate(W.WORKLOADS[1], n=n, dtype=dt)
    mutual_parity(g["pos"], g["mass"], 4, 0.7, leaf)


@pytest.mark.parametrize("theta", [0.05, 0.3, 1.0])
def test_opening_angles_mutual(theta):
    g = W.generate(W.WORKLOADS[2], n=5000)
    mutual_parity(g["pos"], g["mass"], 3, theta, 8)


def test_coincident_particles_mutual():
    """100 coincident points: a depth-21 leaf of more than `leaf` particles, zero separations inside it."""
    rng = np.random.default_rng(0)
    pos = np.vstack([np.full((100, 3), 0.5), rng.random((400, 3))])
    mass = np.full(500, 1.0 / 500)
    mutual_parity(pos, mass, 4, 0.7, 8)


def test_tiny_theta_mutual_equals_direct_sum():
    g = W.generate(W.WORKLOADS[2], n=4000)
    acc, pot, _, _ = gpu_eval(g["pos"], g["mass"], 4, 1e-6, 16, mutual=True)
    acc_d, pot_d = oracle.direct_sum(g["pos"], g["mass"])
    assert accel_error(acc, acc_d).max() < 1e-12
    assert pot_error(pot, pot_d).max() < 1e-12


def test_mutual_deterministic_bitwise():
    g = W.generate(W.WORKLOADS[4], n=50000)
    a1, p1, _, _ = gpu_eval(g["pos"], g["mass"], 4, 0.7, 64, mutual=True)
    a2, p2, _, _ = gpu_eval(g["pos"], g["mass"], 4, 0.7, 64, repeat=3, mutual=True)
    assert np.array_equal(a1, a2) and np.array_equal(p1, p2)


def test_mutual_excludes_rotation():
    from body_forces_morton_b300 import native

    with native.Plan(1000, 4, 0.7, 16, "f32", mutual=True) as pl:
        with pytest.raises(native.FmmError):
            native.fmm_plan_set_m2l_rotation(pl.handle, True)
    with native.Plan(1000, 4, 0.7, 16, "f32", m2l_rotation=True) as pl:
        with pytest.raises(native.FmmError):
            native.fmm_plan_set_mutual(pl.handle, True)


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHILD = r"""
import sys, json, numpy as np, torch
sys.path.insert(0, %r)
from body_forces_morton_b300 import native, workloads as W
g = W.generate(W.WORKLOADS[4], n=20000)
pl = native.Plan(20000, 4, 0.7, 16, "f32", mutual=True)
tp = torch.from_numpy(g["pos"]).cuda(); tm = torch.from_numpy(g["mass"]).cuda()
acc = torch.empty_like(tp)
pl.eval(tp, tm, acc)
np.save(sys.argv[1], acc.cpu().numpy())
print(json.dumps({"retries": pl.stats()["retries"]}))
""" % ROOT


def run_child(fault, out):
    env = dict(os.environ)
    if fault:
        env["BFM_FMM_FAULT"] = fault
    else:
        env.pop("BFM_FMM_FAULT", None)
    r = subprocess.run([sys.executable, "-c", CHILD, str(out)], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_mutual_buffers_regrow_to_the_same_result(tmp_path):
    """Under BFM_FMM_FAULT=capacity the lists and the partner-share buffer start at their minimum; the
    evaluation regrows them and repeats, and the result is the same bit for bit."""
    normal = run_child(None, tmp_path / "n.npy")
    small = run_child("capacity", tmp_path / "s.npy")
    print(f"regrowths: {normal['retries']} normal, {small['retries']} from minimal buffers")
    assert small["retries"] > normal["retries"]
    assert np.array_equal(np.load(tmp_path / "n.npy"), np.load(tmp_path / "s.npy"))


def test_vjp_and_kdk_on_a_mutual_plan():
    """A mutual plan's forward evaluation feeds fmm_vjp and fmm_kdk_step like the default one: the VJP (its
    own stages are the same) agrees with the default plan's to rounding, and so does one KDK step."""
    import torch

    from body_forces_morton_b300 import native

    w = W.WORKLOADS[4]
    n = 40000
    g = W.generate(w, n=n)
    rng = np.random.default_rng(31)
    ab = rng.normal(size=(n, 3)).astype(np.float32)
    pb = rng.normal(size=n).astype(np.float32)
    out = {}
    for mutual in (False, True):
        tp = torch.from_numpy(g["pos"]).cuda()
        tm = torch.from_numpy(g["mass"]).cuda()
        xb = torch.empty_like(tp)
        mb = torch.empty_like(tm)
        vel = torch.zeros_like(tp)
        with native.Plan(n, w.p, w.theta, w.leaf, "f32", mutual=mutual) as pl:
            pl.vjp(tp, tm, torch.from_numpy(ab).cuda(), torch.from_numpy(pb).cuda(), xb, mb)
            torch.cuda.synchronize()
            x2 = tp.clone()
            pl.kdk_step(x2, vel, tm, 1e-3)
            torch.cuda.synchronize()
            out[mutual] = (xb.cpu().numpy(), mb.cpu().numpy(), x2.cpu().numpy(), vel.cpu().numpy())
    d, m = out[False], out[True]
    ex = accel_error(m[0].astype(np.float64), d[0].astype(np.float64))
    ev = accel_error(m[3].astype(np.float64), d[3].astype(np.float64))
    print(f"mutual against default: pos_bar {ex.max():.2e}, KDK velocity {ev.max():.2e}")
    # the VJP's inputs (the forward accelerations, the lists) agree to fp32 rounding, so its outputs do
    # too, up to the cancellation its own fp32 gate allows. The KDK velocity adds the force at the drifted
    # positions, which already differ at the rounding level between the plans, and close pairs amplify
    # that (1 / r^3); each plan's forces are within the parity gate of the oracle, which bounds it
    # (measured 2.8e-5)
    assert ex.max() <= 5e-3 and np.percentile(ex, 99) <= 1e-4
    assert ev.max() <= TOL_ACC["f32"]
    assert np.abs(m[2] - d[2]).max() <= 1e-6 * np.abs(d[2]).max()
