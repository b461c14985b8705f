"""Seeded synthetic particle sets for the FMM workloads.

This module only draws inputs (positions, masses, velocities). It holds none of
the FMM arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from here without sharing any method code.

The five workloads are this library's benchmark configurations (uniform
cube, Plummer spheres, clustered box, KDK run). The pages evaluate none of
them; the jaccpot issue's far-field timings (N = 1e4 and 1e5, theta = 0.7,
order 4, leaf 32) are the context the Plummer sizes echo. All draws use
``numpy.random.default_rng(seed)`` and are fully reproducible.

Recipes (all lengths in the same units, G = 1, total mass 1):

* ``uniform``   -- N points iid uniform in [0, 1)^3, masses 1/N.
* ``plummer``   -- Plummer sphere, scale radius ``a``, truncated at 10a:
  enclosed-mass fraction u ~ U(0, u_max) with u_max = 10^3 / 101^{3/2}
  (the mass fraction inside 10a), radius r = a / sqrt(u^{-2/3} - 1),
  isotropic direction (cos(polar) ~ U(-1, 1), azimuth ~ U(0, 2 pi)),
  centred at the origin, masses 1/N.
* ``clustered`` -- 80 % of the particles in 64 Plummer halos (a = 0.01,
  truncated at 10a, centres iid U[0,1)^3, halo masses log-uniform over two
  decades, i.e. weight 10^{2U}); particle counts proportional to halo mass by
  largest-remainder rounding; the other 20 % uniform in [0, 1)^3; equal
  masses 1/N; the concatenated set is shuffled once.
* velocities    -- each component iid N(0, sigma^2).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PLUMMER_TRUNCATION = 10.0  # truncation radius in units of the scale radius


@dataclass(frozen=True)
class Workload:
    """One named input configuration of the FMM evaluation."""

    name: str
    n: int
    distribution: str  # "uniform" | "plummer" | "clustered"
    dtype: str  # "f32" | "f64"
    p: int
    theta: float
    leaf: int
    seed: int
    velocities: bool = False
    sigma_v: float = 0.0
    notes: str = ""
    extra: dict = field(default_factory=dict)


# The five configurations (index 1..5 == seed).
WORKLOADS = {
    1: Workload("uniform_4096_f64", 4096, "uniform", "f64", 4, 0.7, 32, 1,
                notes="uniform unit cube; checked against oracle FMM and direct sum"),
    2: Workload("plummer_1e4_f64", 10_000, "plummer", "f64", 4, 0.7, 32, 2,
                notes="Plummer a=1 truncated at 10a; one evaluation + stage ms"),
    3: Workload("plummer_1e5_f64", 100_000, "plummer", "f64", 4, 0.7, 32, 3,
                notes="Plummer as above; p/theta sweep vs direct sum on 1000 particles"),
    4: Workload("clustered_2p20_f32", 1 << 20, "clustered", "f32", 4, 0.7, 64, 4,
                notes="64 Plummer halos + 20% background; the N~1e6 throughput point"),
    5: Workload("clustered_2p22_f32_kdk", 1 << 22, "clustered", "f32", 3, 0.6, 64, 5,
                velocities=True, sigma_v=0.1,
                notes="KDK steps; reversibility/momentum run in f64 at N=2^18"),
}

# The fp64 reversibility / momentum companion of workload 5.
KDK_REVERSIBILITY = Workload("clustered_2p18_f64_kdk", 1 << 18, "clustered", "f64", 3, 0.6, 64,
                             5, velocities=True, sigma_v=0.1,
                             notes="20 KDK steps dt=1e-3 forward then 20 backward")


def uniform(n: int, rng: np.random.Generator) -> np.ndarray:
    """n points iid uniform in [0, 1)^3 (float64, shape (n, 3))."""
    return rng.random((n, 3))


def _isotropic(n: int, rng: np.random.Generator) -> np.ndarray:
    cos_t = rng.uniform(-1.0, 1.0, n)
    phi = rng.uniform(0.0, 2.0 * math.pi, n)
    sin_t = np.sqrt(np.maximum(0.0, 1.0 - cos_t * cos_t))
    return np.stack([sin_t * np.cos(phi), sin_t * np.sin(phi), cos_t], axis=1)


def plummer(n: int, rng: np.random.Generator, a: float = 1.0,
            centre=(0.0, 0.0, 0.0)) -> np.ndarray:
    """Plummer sphere of scale radius ``a`` truncated at 10a (float64, (n, 3)).

    Radii by inverting the enclosed-mass fraction u = r^3 / (r^2 + a^2)^{3/2}
    over u in (0, u_max), u_max being the fraction inside the truncation radius.
    """
    rt = PLUMMER_TRUNCATION
    u_max = rt ** 3 / (rt * rt + 1.0) ** 1.5
    u = rng.random(n) * u_max
    with np.errstate(divide="ignore"):
        r = np.where(u > 0.0, a / np.sqrt(np.power(u, -2.0 / 3.0) - 1.0), 0.0)
    return np.asarray(centre, dtype=np.float64)[None, :] + r[:, None] * _isotropic(n, rng)


def largest_remainder(total: int, weights: np.ndarray) -> np.ndarray:
    """Integer counts summing to ``total``, proportional to ``weights``.

    Floors of the exact quotas, then one extra unit to the largest fractional
    remainders (ties go to the lower index).
    """
    w = np.asarray(weights, dtype=np.float64)
    quota = total * w / w.sum()
    base = np.floor(quota).astype(np.int64)
    short = int(total - base.sum())
    if short > 0:
        rem = quota - base
        order = np.lexsort((np.arange(len(w)), -rem))  # largest remainder first
        base[order[:short]] += 1
    return base


def clustered(n: int, rng: np.random.Generator, n_halos: int = 64, a: float = 0.01,
              background_fraction: float = 0.2) -> np.ndarray:
    """Clustered box: 64 Plummer halos plus a 20 % uniform background (float64)."""
    n_bg = int(math.floor(background_fraction * n))
    n_h = n - n_bg
    centres = rng.random((n_halos, 3))
    weights = 10.0 ** (2.0 * rng.random(n_halos))  # log-uniform over two decades
    counts = largest_remainder(n_h, weights)
    parts = [plummer(int(c), rng, a=a, centre=centres[h]) for h, c in enumerate(counts)]
    parts.append(rng.random((n_bg, 3)))
    pos = np.concatenate(parts, axis=0)
    return pos[rng.permutation(n)]


def generate(w: Workload, n: int | None = None, dtype: str | None = None):
    """Positions, masses (and velocities) for workload ``w``.

    ``n`` and ``dtype`` override the workload's own size and precision (used
    for reduced-size parity cases drawn from the same recipe). Returns a dict
    with C-contiguous arrays ``pos`` (n, 3), ``mass`` (n,) and, where the
    workload has them, ``vel`` (n, 3), all of the requested precision.
    """
    n = w.n if n is None else int(n)
    dt = {"f32": np.float32, "f64": np.float64}[w.dtype if dtype is None else dtype]
    rng = np.random.default_rng(w.seed)
    if w.distribution == "uniform":
        pos = uniform(n, rng)
    elif w.distribution == "plummer":
        pos = plummer(n, rng)
    elif w.distribution == "clustered":
        pos = clustered(n, rng)
    else:
        raise ValueError(f"unknown distribution {w.distribution!r}")
    out = {
        "pos": np.ascontiguousarray(pos, dtype=dt),
        "mass": np.full(n, 1.0 / n, dtype=dt),
    }
    if w.velocities:
        out["vel"] = np.ascontiguousarray(rng.normal(0.0, w.sigma_v, (n, 3)), dtype=dt)
    return out


def workload(index_or_name) -> Workload:
    """Look a workload up by its index (1..5) or its name."""
    if isinstance(index_or_name, int):
        return WORKLOADS[index_or_name]
    for w in list(WORKLOADS.values()) + [KDK_REVERSIBILITY]:
        if w.name == index_or_name:
            return w
    raise KeyError(index_or_name)
