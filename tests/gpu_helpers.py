"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare it with the oracle."""
from __future__ import annotations

import numpy as np

STRUCT_INT = ("node_first", "node_count", "node_child0", "node_nchild", "node_parent", "node_level")
TOL_ACC = {"f64": 1e-10, "f32": 1e-4}


def gpu_eval(pos, mass, p, theta, leaf, want_pot=True, exports=(), plan=None, repeat=1, f64_ieee=False,
             m2l_rotation=False, mutual=False):
    """One evaluation through fmm_eval on cuda:0; returns (acc, pot, exports, stats)."""
    import torch

    from body_forces_morton_b300 import native

    dt = "f32" if pos.dtype == np.float32 else "f64"
    n = len(mass)
    own = plan is None
    pl = plan or native.Plan(n, p, theta, leaf, dt, f64_ieee=f64_ieee, m2l_rotation=m2l_rotation, mutual=mutual)
    try:
        tp = torch.from_numpy(np.ascontiguousarray(pos)).cuda()
        tm = torch.from_numpy(np.ascontiguousarray(mass)).cuda()
        acc = torch.empty_like(tp)
        pot = torch.empty_like(tm) if want_pot else None
        for _ in range(repeat):
            pl.eval(tp, tm, acc, pot, stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        ex = {k: pl.export(k) for k in exports}
        st = pl.stats()
        return acc.cpu().numpy(), (pot.cpu().numpy() if want_pot else None), ex, st
    finally:
        if own:
            pl.close()


ALL_STRUCT = ("keys", "perm", "level_off", *STRUCT_INT, "node_lo", "node_hi", "node_centre", "node_half",
              "m2l_off", "m2l_src", "p2p_off", "p2p_src")


def assert_structure_equal(ex, r):
    """Keys, permutation, tree, boxes and lists bit-exact against the oracle."""
    assert np.array_equal(ex["keys"], r.keys), "Morton keys differ"
    assert np.array_equal(ex["perm"].astype(np.int64), r.perm), "sort permutation differs"
    nn = len(r.first)
    assert len(ex["node_first"]) == nn, f"node count {len(ex['node_first'])} != {nn}"
    lo = ex["level_off"][: r.depth + 2].astype(np.int64)
    assert np.array_equal(lo, r.level_off[: r.depth + 2]), "level offsets differ"
    for name, ref in zip(STRUCT_INT, (r.first, r.count, r.child0, r.nchild, r.parent, r.level)):
        assert np.array_equal(ex[name], ref), f"{name} differs"
    for name, ref in (("node_lo", r.lo), ("node_hi", r.hi), ("node_centre", r.centre), ("node_half", r.half)):
        got = ex[name].reshape(nn, 3).astype(np.float64)
        assert np.array_equal(got, ref), f"{name} differs at {np.argwhere(got != ref)[:5].tolist()}"
    for name, ref in (("m2l_off", r.m2l_off), ("p2p_off", r.p2p_off)):
        assert np.array_equal(ex[name].astype(np.int64), ref), f"{name} differs"
    assert np.array_equal(ex["m2l_src"], r.m2l_src), "M2L lists differ"
    assert np.array_equal(ex["p2p_src"], r.p2p_src), "P2P lists differ"


def _weights(r, p):
    """|l|^|n| / n! per node and coefficient (l = the node's half-width vector)."""
    import oracle
    from math import factorial

    mi = oracle.multi_indices(p)
    fact = np.array([factorial(a) * factorial(b) * factorial(c) for a, b, c in mi], dtype=np.float64)
    ln = np.linalg.norm(r.half, axis=1)
    return ln[:, None] ** mi.sum(axis=1)[None, :] / fact[None, :]


def moment_error(got, r, p):
    """max |dM_n| / (M_0 |l|^|n| / n!): the moments' own bound on the node's box."""
    scale = np.abs(r.M[:, :1]) * _weights(r, p) + 1e-300
    return float(np.max(np.abs(got - r.M) / scale))


def local_error(got, ref, r, p):
    """Per node sum_k |dL_k| w_k / sum_k |L_k| w_k with w_k = |l|^|k| / k!: the
    relative size of the polynomial difference on the node's box."""
    w = _weights(r, p)
    den = np.sum(np.abs(ref) * w, axis=1)
    num = np.sum(np.abs(got - ref) * w, axis=1)
    ok = den > 0
    assert np.all(num[~ok] == 0)
    return float(np.max(num[ok] / den[ok])) if ok.any() else 0.0


def accel_error(acc, ref):
    """Per-particle L2 relative error, floored at 1e-3 of the median |a_ref|."""
    na = np.linalg.norm(ref, axis=1)
    floor = 1e-3 * np.median(na[np.isfinite(na)])
    return np.linalg.norm(acc - ref, axis=1) / np.maximum(na, floor)


def pot_error(pot, ref):
    return np.abs(pot - ref) / np.abs(ref)
