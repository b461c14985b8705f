"""CPU oracle for the FMM hot path (test infrastructure).

A plain, slow, fp64 CPU implementation of what one FMM evaluation computes,
written from the JZ-FMM page, plus the exact O(N^2) direct sum. It shares no
code with the CUDA library; only the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import it.

Python side: ctypes marshalling of the C functions in ``fmm_oracle.c``.

Parity of the FMM digits is pinned only through closed forms, invariants and
brute force (the pages print no worked numerical example).
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

DTYPE_F32 = 0
DTYPE_F64 = 1
MAX_DEPTH = 21

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        i64, i32, dbl, vp = C.c_int64, C.c_int, C.c_double, C.c_void_p
        L.orc_ncoef.argtypes = [i32]; L.orc_ncoef.restype = i32
        L.orc_mindex.argtypes = [i32, i32, i32]; L.orc_mindex.restype = i32
        L.orc_direct_sum.argtypes = [i64, vp, vp, i64, vp, vp, vp, i32]
        L.orc_derivs.argtypes = [i32, vp, vp]
        L.orc_p2m.argtypes = [i32, i64, vp, vp, vp, vp]
        L.orc_m2m.argtypes = [i32, vp, vp, vp]
        L.orc_m2l.argtypes = [i32, vp, vp, vp]
        L.orc_l2l.argtypes = [i32, vp, vp, vp]
        L.orc_l2p.argtypes = [i32, vp, vp, vp, vp]
        L.orc_keys.argtypes = [i32, i64, vp, vp, vp]
        L.orc_fmm.argtypes = [i32, i64, vp, vp, i32, dbl, i32, vp, i32, i32, C.POINTER(_Result)]
        L.orc_result_free.argtypes = [C.POINTER(_Result)]
        L.orc_kdk_step.argtypes = [i64, vp, vp, vp, vp, dbl, i32, dbl, i32, i32]
        L.orc_kdk_lattice_step.argtypes = [i64, vp, vp, vp, vp, dbl, i32, i32, i32, dbl, i32, i32]
        L.orc_p2m_dipole.argtypes = [i32, i64, vp, vp, vp, vp, vp]
        L.orc_l2p_hess.argtypes = [i32, vp, vp, vp]
        L.orc_fmm_vjp.argtypes = [i32, i64, vp, vp, vp, vp, i32, dbl, i32, i32, vp, vp]
        for f in ("orc_direct_sum", "orc_derivs", "orc_p2m", "orc_m2m", "orc_m2l", "orc_l2l",
                  "orc_l2p", "orc_keys", "orc_fmm", "orc_kdk_step", "orc_kdk_lattice_step",
                  "orc_p2m_dipole", "orc_l2p_hess", "orc_fmm_vjp"):
            getattr(L, f).restype = i32
        L.orc_result_free.restype = None
        _lib = L
    return _lib


class _Result(C.Structure):
    _fields_ = [
        ("n", C.c_int64), ("n_nodes", C.c_int64), ("n_leaves", C.c_int64),
        ("depth", C.c_int32), ("nc", C.c_int32), ("p", C.c_int32), ("leaf", C.c_int32),
        ("dtype", C.c_int32), ("pad", C.c_int32),
        ("theta", C.c_double),
        ("box", C.c_double * 7),
        ("keys", C.POINTER(C.c_uint64)), ("perm", C.POINTER(C.c_int64)),
        ("level_off", C.c_int64 * (MAX_DEPTH + 2)),
        ("first", C.POINTER(C.c_int32)), ("count", C.POINTER(C.c_int32)),
        ("child0", C.POINTER(C.c_int32)), ("nchild", C.POINTER(C.c_int32)),
        ("parent", C.POINTER(C.c_int32)), ("level", C.POINTER(C.c_int32)),
        ("lo", C.POINTER(C.c_double)), ("hi", C.POINTER(C.c_double)),
        ("centre", C.POINTER(C.c_double)), ("half", C.POINTER(C.c_double)),
        ("M", C.POINTER(C.c_double)), ("Lm2l", C.POINTER(C.c_double)), ("L", C.POINTER(C.c_double)),
        ("n_m2l_pairs", C.c_int64), ("n_p2p_pairs", C.c_int64),
        ("n_m2l", C.c_int64), ("n_p2p", C.c_int64),
        ("m2l_off", C.POINTER(C.c_int64)), ("m2l_src", C.POINTER(C.c_int32)),
        ("p2p_off", C.POINTER(C.c_int64)), ("p2p_src", C.POINTER(C.c_int32)),
        ("n_p2p_interactions", C.c_int64),
        ("acc", C.POINTER(C.c_double)), ("pot", C.POINTER(C.c_double)),
        ("t_stage", C.c_double * 8),
    ]


STAGES = ("keys_sort", "tree", "upward", "walk", "m2l", "l2l", "leaf", "total")


def _ptr(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def _check(st, what):
    if st != 0:
        raise RuntimeError(f"oracle {what} failed with status {st}")


def ncoef(p: int) -> int:
    return int(lib().orc_ncoef(p))


def mindex(nx: int, ny: int, nz: int) -> int:
    return int(lib().orc_mindex(nx, ny, nz))


def multi_indices(p: int) -> np.ndarray:
    """(ncoef, 3) table of exponents in the coefficient order."""
    out = np.zeros((ncoef(p), 3), dtype=np.int64)
    for d in range(p + 1):
        for nx in range(d, -1, -1):
            for ny in range(d - nx, -1, -1):
                out[mindex(nx, ny, d - nx - ny)] = (nx, ny, d - nx - ny)
    return out


def direct_sum(pos, mass, targets=None, nthreads: int = 0):
    """Exact O(N^2) fp64 sum (compensated); returns (acc (n,3), pot (n,)).

    With ``targets`` (indices) only those rows are computed; the other rows
    are NaN.
    """
    pos = np.ascontiguousarray(pos, dtype=np.float64)
    mass = np.ascontiguousarray(mass, dtype=np.float64)
    n = len(mass)
    acc = np.full((n, 3), np.nan)
    pot = np.full(n, np.nan)
    t = None if targets is None else np.ascontiguousarray(targets, dtype=np.int64)
    _check(lib().orc_direct_sum(n, _ptr(pos), _ptr(mass), 0 if t is None else len(t), _ptr(t),
                                _ptr(acc), _ptr(pot), nthreads), "direct_sum")
    return acc, pot


def derivs(p: int, R) -> np.ndarray:
    R = np.ascontiguousarray(R, dtype=np.float64)
    D = np.zeros(ncoef(p))
    _check(lib().orc_derivs(p, _ptr(R), _ptr(D)), "derivs")
    return D


def p2m(p: int, pos, mass, c) -> np.ndarray:
    pos = np.ascontiguousarray(pos, dtype=np.float64).reshape(-1, 3)
    mass = np.ascontiguousarray(mass, dtype=np.float64)
    c = np.ascontiguousarray(c, dtype=np.float64)
    M = np.zeros(ncoef(p))
    _check(lib().orc_p2m(p, len(mass), _ptr(pos), _ptr(mass), _ptr(c), _ptr(M)), "p2m")
    return M


def m2m(p: int, Mc, d) -> np.ndarray:
    Mc = np.ascontiguousarray(Mc, dtype=np.float64)
    d = np.ascontiguousarray(d, dtype=np.float64)
    Mp = np.zeros(ncoef(p))
    _check(lib().orc_m2m(p, _ptr(Mc), _ptr(d), _ptr(Mp)), "m2m")
    return Mp


def m2l(p: int, M, R) -> np.ndarray:
    M = np.ascontiguousarray(M, dtype=np.float64)
    R = np.ascontiguousarray(R, dtype=np.float64)
    L = np.zeros(ncoef(p))
    _check(lib().orc_m2l(p, _ptr(M), _ptr(R), _ptr(L)), "m2l")
    return L


def l2l(p: int, Lp, e) -> np.ndarray:
    Lp = np.ascontiguousarray(Lp, dtype=np.float64)
    e = np.ascontiguousarray(e, dtype=np.float64)
    Lc = np.zeros(ncoef(p))
    _check(lib().orc_l2l(p, _ptr(Lp), _ptr(e), _ptr(Lc)), "l2l")
    return Lc


def p2m_dipole(p: int, pos, q, d, c) -> np.ndarray:
    """Moments of sources with monopoles q (None = 0) and dipoles d [n x 3] about c."""
    pos = np.ascontiguousarray(pos, dtype=np.float64).reshape(-1, 3)
    d = np.ascontiguousarray(d, dtype=np.float64).reshape(-1, 3)
    qq = None if q is None else np.ascontiguousarray(q, dtype=np.float64)
    c = np.ascontiguousarray(c, dtype=np.float64)
    M = np.zeros(ncoef(p))
    _check(lib().orc_p2m_dipole(p, len(pos), _ptr(pos), _ptr(qq), _ptr(d), _ptr(c), _ptr(M)), "p2m_dipole")
    return M


def l2p_hess(p: int, L, dx) -> np.ndarray:
    """Hessian (xx, xy, xz, yy, yz, zz) of the local series L at offset dx."""
    L = np.ascontiguousarray(L, dtype=np.float64)
    dx = np.ascontiguousarray(dx, dtype=np.float64)
    H = np.zeros(6)
    _check(lib().orc_l2p_hess(p, _ptr(L), _ptr(dx), _ptr(H)), "l2p_hess")
    return H


def l2p(p: int, L, dx):
    """Potential and acceleration of the local series L at offset dx."""
    L = np.ascontiguousarray(L, dtype=np.float64)
    dx = np.ascontiguousarray(dx, dtype=np.float64)
    pot = np.zeros(1)
    acc = np.zeros(3)
    _check(lib().orc_l2p(p, _ptr(L), _ptr(dx), _ptr(pot), _ptr(acc)), "l2p")
    return float(pot[0]), acc


def keys(pos):
    """Morton keys in the caller's order and the root box (lo[3], hi[3], side)."""
    pos = np.ascontiguousarray(pos)
    dt = DTYPE_F32 if pos.dtype == np.float32 else DTYPE_F64
    if pos.dtype not in (np.float32, np.float64):
        raise TypeError("pos must be float32 or float64")
    k = np.zeros(len(pos), dtype=np.uint64)
    box = np.zeros(7)
    _check(lib().orc_keys(dt, len(pos), _ptr(pos), _ptr(k), _ptr(box)), "keys")
    return k, box


@dataclass
class FmmResult:
    n: int
    p: int
    theta: float
    leaf: int
    dtype: str
    depth: int
    box: np.ndarray
    keys: np.ndarray
    perm: np.ndarray
    level_off: np.ndarray
    first: np.ndarray
    count: np.ndarray
    child0: np.ndarray
    nchild: np.ndarray
    parent: np.ndarray
    level: np.ndarray
    lo: np.ndarray
    hi: np.ndarray
    centre: np.ndarray
    half: np.ndarray
    M: np.ndarray | None
    Lm2l: np.ndarray | None
    L: np.ndarray | None
    n_m2l_pairs: int
    n_p2p_pairs: int
    m2l_off: np.ndarray
    m2l_src: np.ndarray
    p2p_off: np.ndarray
    p2p_src: np.ndarray
    n_p2p_interactions: int
    acc: np.ndarray | None
    pot: np.ndarray | None
    t_stage: dict

    @property
    def n_nodes(self) -> int:
        return len(self.first)

    def m2l_list(self, a: int) -> np.ndarray:
        return self.m2l_src[self.m2l_off[a]:self.m2l_off[a + 1]]

    def p2p_list(self, a: int) -> np.ndarray:
        return self.p2p_src[self.p2p_off[a]:self.p2p_off[a + 1]]


def _arr(ptr, n, dtype):
    if n == 0 or not ptr:
        return np.zeros(0, dtype=dtype)
    return np.ctypeslib.as_array(ptr, shape=(n,)).astype(dtype, copy=True)


def fmm(pos, mass, p: int = 4, theta: float = 0.7, leaf: int = 32, eval_mask=None,
        tree_only: bool = False, nthreads: int = 0) -> FmmResult:
    """One oracle FMM evaluation (inputs float32 or float64, same dtype).

    ``eval_mask`` (bool array over particles) restricts the evaluation to the
    flagged particles; ``tree_only`` stops after the walk.
    """
    pos = np.ascontiguousarray(pos)
    mass = np.ascontiguousarray(mass)
    if pos.dtype != mass.dtype or pos.dtype not in (np.float32, np.float64):
        raise TypeError("pos and mass must share a float32/float64 dtype")
    dt = DTYPE_F32 if pos.dtype == np.float32 else DTYPE_F64
    n = len(mass)
    mask = None if eval_mask is None else np.ascontiguousarray(eval_mask, dtype=np.uint8)
    r = _Result()
    st = lib().orc_fmm(dt, n, _ptr(pos), _ptr(mass), p, float(theta), leaf, _ptr(mask),
                       1 if tree_only else 0, nthreads, C.byref(r))
    _check(st, "fmm")
    try:
        nn = r.n_nodes
        nc = r.nc
        out = FmmResult(
            n=n, p=p, theta=theta, leaf=leaf, dtype="f32" if dt == DTYPE_F32 else "f64",
            depth=r.depth, box=np.array(r.box[:]),
            keys=_arr(r.keys, n, np.uint64), perm=_arr(r.perm, n, np.int64),
            level_off=np.array(r.level_off[:], dtype=np.int64),
            first=_arr(r.first, nn, np.int32), count=_arr(r.count, nn, np.int32),
            child0=_arr(r.child0, nn, np.int32), nchild=_arr(r.nchild, nn, np.int32),
            parent=_arr(r.parent, nn, np.int32), level=_arr(r.level, nn, np.int32),
            lo=_arr(r.lo, 3 * nn, np.float64).reshape(nn, 3),
            hi=_arr(r.hi, 3 * nn, np.float64).reshape(nn, 3),
            centre=_arr(r.centre, 3 * nn, np.float64).reshape(nn, 3),
            half=_arr(r.half, 3 * nn, np.float64).reshape(nn, 3),
            M=None if tree_only else _arr(r.M, nn * nc, np.float64).reshape(nn, nc),
            Lm2l=None if tree_only else _arr(r.Lm2l, nn * nc, np.float64).reshape(nn, nc),
            L=None if tree_only else _arr(r.L, nn * nc, np.float64).reshape(nn, nc),
            n_m2l_pairs=r.n_m2l_pairs, n_p2p_pairs=r.n_p2p_pairs,
            m2l_off=_arr(r.m2l_off, nn + 1, np.int64), m2l_src=_arr(r.m2l_src, r.n_m2l, np.int32),
            p2p_off=_arr(r.p2p_off, nn + 1, np.int64), p2p_src=_arr(r.p2p_src, r.n_p2p, np.int32),
            n_p2p_interactions=r.n_p2p_interactions,
            acc=None if tree_only else _arr(r.acc, 3 * n, np.float64).reshape(n, 3),
            pot=None if tree_only else _arr(r.pot, n, np.float64),
            t_stage=dict(zip(STAGES, r.t_stage[:])),
        )
    finally:
        lib().orc_result_free(C.byref(r))
    return out


def fmm_vjp(pos, mass, acc_bar, pot_bar=None, p: int = 4, theta: float = 0.7, leaf: int = 32, nthreads: int = 0):
    """Vector-Jacobian product of one FMM evaluation (see orc_fmm_vjp): returns (pos_bar [n x 3],
    mass_bar [n]) for the cotangents acc_bar [n x 3] and pot_bar [n] (or None), in fp64."""
    pos = np.ascontiguousarray(pos)
    mass = np.ascontiguousarray(mass)
    if pos.dtype != mass.dtype or pos.dtype not in (np.float32, np.float64):
        raise TypeError("pos and mass must share a float32/float64 dtype")
    dt = DTYPE_F32 if pos.dtype == np.float32 else DTYPE_F64
    ab = np.ascontiguousarray(acc_bar, dtype=np.float64).reshape(-1, 3)
    pb = None if pot_bar is None else np.ascontiguousarray(pot_bar, dtype=np.float64)
    n = len(mass)
    xb = np.zeros((n, 3))
    mb = np.zeros(n)
    _check(lib().orc_fmm_vjp(dt, n, _ptr(pos), _ptr(mass), _ptr(ab), _ptr(pb), p, float(theta), leaf, nthreads,
                             _ptr(xb), _ptr(mb)), "fmm_vjp")
    return xb, mb


def kdk_step(pos, vel, mass, acc, dt: float, p: int, theta: float, leaf: int, nthreads: int = 0):
    """One fp64 kick-drift-kick step in place; ``acc`` must hold a(pos) on entry."""
    for a in (pos, vel, mass, acc):
        if a.dtype != np.float64 or not a.flags.c_contiguous:
            raise TypeError("kdk_step works on C-contiguous float64 arrays")
    _check(lib().orc_kdk_step(len(mass), _ptr(pos), _ptr(vel), _ptr(mass), _ptr(acc), float(dt), p,
                              float(theta), leaf, nthreads), "kdk_step")


def kdk_lattice_step(pos, vel, mass, acc, dt: float, pos_exp: int, vel_exp: int, p: int, theta: float, leaf: int,
                     nthreads: int = 0):
    """One lattice kick-drift-kick step in place (fp64); see orc_kdk_lattice_step."""
    for a in (pos, vel, mass, acc):
        if a.dtype != np.float64 or not a.flags.c_contiguous:
            raise TypeError("kdk_lattice_step works on C-contiguous float64 arrays")
    _check(lib().orc_kdk_lattice_step(len(mass), _ptr(pos), _ptr(vel), _ptr(mass), _ptr(acc), float(dt), pos_exp,
                                      vel_exp, p, float(theta), leaf, nthreads), "kdk_lattice_step")
