"""Checks of the seeded input generators (recipes stated in the workloads module)."""
import numpy as np
from scipy import stats

from body_forces_morton_b300 import workloads as W


def test_plummer_radial_profile():
    """Radii follow the truncated Plummer enclosed-mass law r^3/(r^2+a^2)^{3/2} (KS test)."""
    g = W.generate(W.WORKLOADS[2])
    r = np.linalg.norm(g["pos"], axis=1)
    u_max = 1000.0 / 101.0 ** 1.5
    cdf = lambda x: (x ** 3 / (x * x + 1.0) ** 1.5) / u_max
    assert r.max() <= 10.0 + 1e-12
    assert stats.kstest(r, cdf).pvalue > 1e-3
    # isotropy: mean direction near zero
    assert np.linalg.norm((g["pos"] / r[:, None]).mean(axis=0)) < 0.05


def test_clustered_recipe():
    n = 1 << 16
    g = W.generate(W.WORKLOADS[4], n=n)
    assert g["pos"].dtype == np.float32 and g["pos"].shape == (n, 3)
    assert np.all(g["mass"] == np.float32(1.0 / n))
    w = np.array([1.0, 3.0, 6.0])
    assert list(W.largest_remainder(10, w)) == [1, 3, 6]
    assert W.largest_remainder(7, np.array([1.0, 1.0, 1.0])).tolist() == [3, 2, 2]
    # 20% of the particles are background in the unit cube; halos are compact
    inside = np.all((g["pos"] >= 0) & (g["pos"] < 1), axis=1)
    assert inside.mean() > 0.8


def test_reproducible_and_sized():
    a = W.generate(W.WORKLOADS[1])
    b = W.generate(W.WORKLOADS[1])
    assert np.array_equal(a["pos"], b["pos"]) and a["pos"].shape == (4096, 3)
    assert np.all((a["pos"] >= 0) & (a["pos"] < 1))
    v = W.generate(W.KDK_REVERSIBILITY, n=50000)
    assert abs(v["vel"].std() - 0.1) < 0.002
    assert v["pos"].dtype == np.float64
