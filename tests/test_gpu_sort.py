"""The radix sort's dispatch edges against the oracle's keys and a stable sort.

The evaluation sorts (key, index) pairs by the keys' high words with one
cooperative launch for the radix passes when the tiles number at least 16 and
all fit on the GPU at once, and with one kernel per pass otherwise (2^19
switches the tile from 2048 to 4096 keys); runs of equal high words are then
sorted by low word and index, by one thread up to 32 keys, by a block in
shared memory up to 4096 and by a block's four stable passes beyond (after an
evaluation with many keys in long runs the plan sorts all 8 digits). Each case
checks the sorted keys and the permutation bit for bit against the oracle's
keys sorted by (key, index), with coincident particles so that equal keys must
keep their index order.
"""
import numpy as np
import pytest

import oracle
from body_forces_morton_b300 import workloads as W
from gpu_helpers import gpu_eval

pytestmark = pytest.mark.gpu

# 15 tiles of 2048 (per pass), 16 (cooperative), 256 tiles of 2048 and 128 of 4096 (cooperative),
# about 500 tiles of 4096 (more than fit at once: per pass)
SIZES = [15 * 2048, 15 * 2048 + 1, (1 << 19) - 1, 1 << 19, 2_100_000]


@pytest.mark.parametrize("n", SIZES)
def test_sort_dispatch_edges(n):
    g = W.generate(W.WORKLOADS[4], n=n)
    pos = np.array(g["pos"])
    pos[100:300] = pos[100]  # 200 equal keys
    k, _ = oracle.keys(pos)
    perm = np.lexsort((np.arange(n), k))
    _, _, ex, _ = gpu_eval(pos, g["mass"], 0, 0.7, 64, want_pot=False, exports=("keys", "perm"))
    assert np.array_equal(ex["keys"], k[perm]), "sorted keys differ"
    assert np.array_equal(ex["perm"].astype(np.int64), perm), "sort permutation differs"


@pytest.mark.parametrize("repeat", [1, 2])
def test_sort_long_runs(repeat):
    """Runs of equal high key words of 40 and 3000 coincident particles and of 6000 particles in one
    cube of side 2^-14 of the box (distinct low words): the warp path and both block paths (shared memory,
    passes). These runs hold far more than 1/64 of the keys, so a second evaluation on the same plan sorts
    all 8 digits instead; both give the same order."""
    rng = np.random.default_rng(7)
    bg = rng.random((30000, 3))
    cube = 0.3 + rng.random((6000, 3)) * 2.0 ** -14
    pos = np.vstack([bg, cube, np.full((3000, 3), 0.6), np.full((40, 3), 0.7)])
    pos = pos[rng.permutation(len(pos))]
    n = len(pos)
    mass = np.full(n, 1.0 / n)
    k, _ = oracle.keys(pos)
    perm = np.lexsort((np.arange(n), k))
    hi = k[perm] >> np.uint64(32)
    runs = np.diff(np.flatnonzero(np.concatenate([[True], hi[1:] != hi[:-1], [True]])))
    assert runs.max() > 4096 and ((runs > 32) & (runs <= 4096)).sum() >= 2
    _, _, ex, _ = gpu_eval(pos, mass, 0, 0.7, 64, want_pot=False, exports=("keys", "perm"), repeat=repeat)
    assert np.array_equal(ex["keys"], k[perm]), "sorted keys differ"
    assert np.array_equal(ex["perm"].astype(np.int64), perm), "sort permutation differs"

