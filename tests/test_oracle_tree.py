"""Pins of the oracle's keys, sort, octree and dual-tree walk.

The integer structure must be exactly right, so it is checked against an
independent numpy computation of the Morton keys (bit spreading instead of a
bit loop; numpy's stable argsort instead of the C sort) and against the
structural invariants the JZ-FMM page states ("Why this works well on GPUs":
neighbouring particles and child nodes contiguous) and the walk's contract
(every ordered particle pair covered exactly once; the opening criterion
eq. decides acceptance).
"""
import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W


def spread3(v):
    """Spread the low 21 bits of v so bit b lands at 3b (magic-number method)."""
    v = v.astype(np.uint64) & np.uint64(0x1FFFFF)
    v = (v | (v << np.uint64(32))) & np.uint64(0x1F00000000FFFF)
    v = (v | (v << np.uint64(16))) & np.uint64(0x1F0000FF0000FF)
    v = (v | (v << np.uint64(8))) & np.uint64(0x100F00F00F00F00F)
    v = (v | (v << np.uint64(4))) & np.uint64(0x10C30C30C30C30C3)
    v = (v | (v << np.uint64(2))) & np.uint64(0x1249249249249249)
    return v


def numpy_keys(pos):
    lo = pos.min(axis=0)
    hi = pos.max(axis=0)
    ext = hi - lo
    side = ext.max()
    if not side > 0:
        side = pos.dtype.type(1)
    q = np.floor(((pos - lo) / side) * pos.dtype.type(2097152.0))
    q = np.minimum(q.astype(np.int64), 2097151).astype(np.uint64)
    return (spread3(q[:, 0]) << np.uint64(2)) | (spread3(q[:, 1]) << np.uint64(1)) | spread3(q[:, 2])


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_keys_match_independent_numpy(cfg, dtype):
    g = W.generate(W.WORKLOADS[cfg], n=20000, dtype=dtype)
    k, box = oracle.keys(g["pos"])
    assert np.array_equal(k, numpy_keys(g["pos"]))
    assert box[6] == (g["pos"].max(axis=0) - g["pos"].min(axis=0)).max()


def test_degenerate_extent_keys():
    pos = np.full((10, 3), 0.25)
    k, box = oracle.keys(pos)
    assert box[6] == 1.0 and np.all(k == 0)
    r = oracle.fmm(pos, np.full(10, 0.1), 4, 0.7, 4, tree_only=True)
    # ten coincident points: one chain down to depth 21, which may exceed the leaf size
    assert r.depth == 21 and r.count[-1] == 10


def check_tree(r, pos):
    n = r.n
    nn = r.n_nodes
    # sort: stable by key, perm a permutation
    assert np.array_equal(np.sort(r.perm), np.arange(n))
    k_unsorted, _ = oracle.keys(pos)
    order = np.argsort(k_unsorted, kind="stable")
    assert np.array_equal(order, r.perm)
    assert np.array_equal(k_unsorted[order], r.keys)
    # root and breadth-first order
    assert r.first[0] == 0 and r.count[0] == n and r.parent[0] == -1 and r.level[0] == 0
    assert np.all(np.diff(r.level) >= 0)
    for l in range(r.depth + 1):
        a, b = r.level_off[l], r.level_off[l + 1]
        assert np.all(r.level[a:b] == l)
        assert np.all(np.diff(r.first[a:b]) > 0)
    for a in range(nn):
        is_leaf = r.nchild[a] == 0
        assert is_leaf == (r.count[a] <= r.leaf or r.level[a] == 21)
        if not is_leaf:
            ch = np.arange(r.child0[a], r.child0[a] + r.nchild[a])
            assert np.all(r.parent[ch] == a) and np.all(r.level[ch] == r.level[a] + 1)
            assert r.first[ch[0]] == r.first[a]
            assert np.all(r.first[ch[1:]] == r.first[ch[:-1]] + r.count[ch[:-1]])
            assert r.count[ch].sum() == r.count[a] and np.all(r.count[ch] > 0)
        # all particles of a node share its Morton prefix, siblings differ
        shift = np.uint64(3 * (21 - r.level[a]))
        seg = r.keys[r.first[a]:r.first[a] + r.count[a]] >> shift
        assert np.all(seg == seg[0])
        # tight box, centre and half-width in the input precision
        xs = pos[r.perm[r.first[a]:r.first[a] + r.count[a]]]
        assert np.array_equal(r.lo[a], xs.min(axis=0).astype(np.float64))
        assert np.array_equal(r.hi[a], xs.max(axis=0).astype(np.float64))
        t = pos.dtype.type
        assert np.array_equal(r.centre[a], ((xs.min(axis=0) + xs.max(axis=0)) * t(0.5)).astype(np.float64))
        assert np.array_equal(r.half[a], ((xs.max(axis=0) - xs.min(axis=0)) * t(0.5)).astype(np.float64))


@pytest.mark.parametrize("cfg,n,leaf,dtype", [(1, 3000, 32, "f64"), (2, 5000, 16, "f64"),
                                              (4, 8000, 64, "f32"), (4, 3000, 8, "f64")])
def test_tree_invariants(cfg, n, leaf, dtype):
    g = W.generate(W.WORKLOADS[cfg], n=n, dtype=dtype)
    r = oracle.fmm(g["pos"], g["mass"], 4, 0.7, leaf, tree_only=True)
    check_tree(r, g["pos"])


def ordered_pair_cover(r):
    """Count, for every ordered particle pair (i, j) in sorted order, how many
    list entries cover it (M2L A<-B or P2P A<-B with i in A, j in B)."""
    n = r.n
    cover = np.zeros((n, n), dtype=np.int32)
    for off, src in ((r.m2l_off, r.m2l_src), (r.p2p_off, r.p2p_src)):
        for a in range(r.n_nodes):
            ia = slice(r.first[a], r.first[a] + r.count[a])
            for b in src[off[a]:off[a + 1]]:
                cover[ia, r.first[b]:r.first[b] + r.count[b]] += 1
    return cover


def accepted(r, a, b):
    t = np.float32 if r.dtype == "f32" else np.float64
    la, lb = r.half[a].astype(t), r.half[b].astype(t)
    ca, cb = r.centre[a].astype(t), r.centre[b].astype(t)
    s = la + lb
    d = ca - cb
    s2 = (s[0] * s[0] + s[1] * s[1]) + s[2] * s[2]
    r2 = (d[0] * d[0] + d[1] * d[1]) + d[2] * d[2]
    return bool(s2 < t(r.theta * r.theta) * r2)


@pytest.mark.parametrize("n,leaf,theta,dtype", [(2, 1, 0.5, "f64"), (7, 1, 0.3, "f64"), (33, 2, 0.7, "f64"),
                                                 (64, 4, 0.5, "f32"), (64, 1, 0.7, "f64"),
                                                 (1500, 8, 0.7, "f64"), (1500, 16, 0.4, "f32")])
def test_walk_covers_every_pair_exactly_once(n, leaf, theta, dtype):
    g = W.generate(W.WORKLOADS[2], n=n, dtype=dtype)
    r = oracle.fmm(g["pos"], g["mass"], 3, theta, leaf, tree_only=True)
    cover = ordered_pair_cover(r)
    assert np.all(cover == 1)
    # lists are symmetric, sorted by (receiver, source), and follow the criterion
    for off, src, m2l in ((r.m2l_off, r.m2l_src, True), (r.p2p_off, r.p2p_src, False)):
        pairs = {(a, int(b)) for a in range(r.n_nodes) for b in src[off[a]:off[a + 1]]}
        assert all((b, a) in pairs for a, b in pairs)
        for a in range(r.n_nodes):
            seg = src[off[a]:off[a + 1]]
            assert np.all(np.diff(seg) > 0)
        for a, b in pairs:
            if m2l:
                assert a != b and accepted(r, a, b)
            else:
                assert r.nchild[a] == 0 and r.nchild[b] == 0
                assert a == b or not accepted(r, a, b)
    assert r.n_p2p_interactions == sum(
        r.count[a] * r.count[b] for a in range(r.n_nodes) for b in r.p2p_src[r.p2p_off[a]:r.p2p_off[a + 1]])


def test_tiny_theta_accepts_only_point_pairs():
    """As theta -> 0 only pairs of zero-extent nodes (single particles) pass the criterion."""
    g = W.generate(W.WORKLOADS[1], n=2000)
    r = oracle.fmm(g["pos"], g["mass"], 4, 1e-6, 16, tree_only=True)
    for a in range(r.n_nodes):
        for b in r.m2l_list(a):
            assert np.all(r.half[a] == 0) and np.all(r.half[b] == 0)
    n_m2l_particle_pairs = sum(r.count[a] * r.count[b] for a in range(r.n_nodes) for b in r.m2l_list(a))
    assert r.n_p2p_interactions + n_m2l_particle_pairs == 2000 * 2000
