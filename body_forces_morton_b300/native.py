"""Thin ctypes binding of ``libbfm_fmm.so`` (declared in ``include/fmm.h``).

The functions keep the C names and only marshal arguments; every step of an
evaluation runs in the library's CUDA kernels. Tensor arguments may be
``torch.Tensor`` (device tensors for ``fmm_eval``/``fmm_kdk_step``, host
tensors for ``fmm_eval_host``), numpy arrays (host) or raw integer pointers.
There is no fallback: a missing library raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libbfm_fmm.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "fmm.h")

FMM_F32, FMM_F64 = 0, 1
STATUS = {0: "FMM_OK", 1: "FMM_ERR_INVALID_ARG", 2: "FMM_ERR_OOM", 3: "FMM_ERR_CUDA", 4: "FMM_ERR_CAPACITY",
          5: "FMM_ERR_NONFINITE", 6: "FMM_ERR_INTERNAL"}
STAGES = ("keys", "sort", "tree", "upward", "walk", "lists", "m2l", "l2l", "l2p", "p2p")
N_STAGES = len(STAGES)

EXPORTS = {
    "keys": (0, np.uint64), "perm": (1, np.uint32), "node_first": (2, np.int32), "node_count": (3, np.int32),
    "node_child0": (4, np.int32), "node_nchild": (5, np.int32), "node_parent": (6, np.int32),
    "node_level": (7, np.int32), "level_off": (8, np.int32), "node_lo": (9, None), "node_hi": (10, None),
    "node_centre": (11, None), "node_half": (12, None), "multipole": (13, None), "local_m2l": (14, None),
    "local": (15, None), "m2l_off": (16, np.int32), "m2l_src": (17, np.int32), "p2p_off": (18, np.int32),
    "p2p_src": (19, np.int32),
}


class FmmError(RuntimeError):
    """A library call returned a status other than FMM_OK."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class fmm_stats(C.Structure):
    _fields_ = [
        ("n", C.c_int64), ("n_nodes", C.c_int64), ("n_leaves", C.c_int64),
        ("depth", C.c_int32), ("p", C.c_int32),
        ("n_m2l", C.c_int64), ("n_p2p", C.c_int64), ("n_p2p_interactions", C.c_int64),
        ("walk_pairs", C.c_int64),
        ("stage_ms", C.c_double * N_STAGES), ("total_ms", C.c_double),
        ("launches", C.c_int32), ("retries", C.c_int32),
    ]


_lib = None


def declared_functions(header: str = HEADER):
    """Names of the functions ``include/fmm.h`` declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fmm_[a-z_]+)\s*\(", text)))


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing (run body_forces_morton_b300/build.py)")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64, dbl = C.c_void_p, C.c_int, C.c_int64, C.c_double
        L.fmm_plan_create.argtypes = [i64, i32, dbl, i32, i32]
        L.fmm_plan_create.restype = vp
        L.fmm_eval.argtypes = [vp, vp, vp, vp, vp, vp]
        L.fmm_eval_host.argtypes = [vp, vp, vp, vp, vp, vp]
        L.fmm_kdk_step.argtypes = [vp, vp, vp, vp, dbl, vp]
        L.fmm_kdk_step_lattice.argtypes = [vp, vp, vp, vp, dbl, i32, i32, vp]
        L.fmm_kdk_reset.argtypes = [vp]
        L.fmm_kdk_reset.restype = None
        L.fmm_destroy.argtypes = [vp]
        L.fmm_destroy.restype = None
        L.fmm_last_error.argtypes = []
        L.fmm_last_error.restype = C.c_char_p
        L.fmm_plan_stats.argtypes = [vp, C.POINTER(fmm_stats)]
        L.fmm_plan_export_size.argtypes = [vp, i32]
        L.fmm_plan_export_size.restype = i64
        L.fmm_plan_export.argtypes = [vp, i32, vp, i64]
        L.fmm_morton_keys_noalloc.argtypes = [vp, i64, i32, vp, vp, vp]
        L.fmm_vjp.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        L.fmm_plan_set_f64_ieee.argtypes = [vp, i32]
        L.fmm_plan_set_m2l_rotation.argtypes = [vp, i32]
        L.fmm_plan_set_mutual.argtypes = [vp, i32]
        for f in ("fmm_eval", "fmm_eval_host", "fmm_kdk_step", "fmm_kdk_step_lattice", "fmm_plan_stats", "fmm_plan_export",
                  "fmm_morton_keys_noalloc", "fmm_vjp", "fmm_plan_set_f64_ieee", "fmm_plan_set_m2l_rotation",
                  "fmm_plan_set_mutual"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        if not x.flags.c_contiguous:
            raise ValueError("array arguments must be C-contiguous")
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


def _check(status):
    if status != 0:
        raise FmmError(status, fmm_last_error())


def fmm_last_error() -> str:
    return lib().fmm_last_error().decode()


def fmm_plan_create(n: int, p: int, theta: float, leaf: int, dtype: int):
    h = lib().fmm_plan_create(int(n), int(p), float(theta), int(leaf), int(dtype))
    if not h:
        raise FmmError(1, fmm_last_error())
    return h


def fmm_eval(plan, pos, mass, acc_out, pot_out=None, stream=None):
    _check(lib().fmm_eval(plan, _ptr(pos), _ptr(mass), _ptr(acc_out), _ptr(pot_out), _stream(stream)))


def fmm_eval_host(plan, pos, mass, acc_out, pot_out=None, stream=None):
    _check(lib().fmm_eval_host(plan, _ptr(pos), _ptr(mass), _ptr(acc_out), _ptr(pot_out), _stream(stream)))


def fmm_kdk_step(plan, pos, vel, mass, dt: float, stream=None):
    _check(lib().fmm_kdk_step(plan, _ptr(pos), _ptr(vel), _ptr(mass), float(dt), _stream(stream)))


def fmm_kdk_step_lattice(plan, pos, vel, mass, dt: float, pos_exp: int, vel_exp: int, stream=None):
    _check(lib().fmm_kdk_step_lattice(plan, _ptr(pos), _ptr(vel), _ptr(mass), float(dt), int(pos_exp), int(vel_exp),
                                      _stream(stream)))


def fmm_plan_set_f64_ieee(plan, on: bool):
    _check(lib().fmm_plan_set_f64_ieee(plan, 1 if on else 0))


def fmm_plan_set_m2l_rotation(plan, on: bool):
    _check(lib().fmm_plan_set_m2l_rotation(plan, 1 if on else 0))


def fmm_plan_set_mutual(plan, on: bool):
    _check(lib().fmm_plan_set_mutual(plan, 1 if on else 0))


def fmm_vjp(plan, pos, mass, acc_bar, pot_bar, pos_bar, mass_bar, stream=None):
    _check(lib().fmm_vjp(plan, _ptr(pos), _ptr(mass), _ptr(acc_bar), _ptr(pot_bar), _ptr(pos_bar), _ptr(mass_bar),
                         _stream(stream)))


def fmm_morton_keys_noalloc(pos, n: int, dtype: int, keys_out, box_out=None, stream=None):
    """Root box and Morton keys of n <= 2^21 particles with no device allocation."""
    st = lib().fmm_morton_keys_noalloc(_ptr(pos), int(n), int(dtype), _ptr(keys_out), _ptr(box_out),
                                       _stream(stream))
    if st != 0:
        raise FmmError(st, "fmm_morton_keys_noalloc failed")


def fmm_kdk_reset(plan):
    lib().fmm_kdk_reset(plan)


def fmm_destroy(plan):
    lib().fmm_destroy(plan)


def fmm_plan_stats(plan) -> dict:
    s = fmm_stats()
    _check(lib().fmm_plan_stats(plan, C.byref(s)))
    d = {f: getattr(s, f) for f, _ in fmm_stats._fields_ if f != "stage_ms"}
    d["stage_ms"] = dict(zip(STAGES, s.stage_ms[:]))
    return d


def fmm_plan_export(plan, what: str, dtype=None) -> np.ndarray:
    """Copy an internal array of the last evaluation to a numpy array.

    ``dtype`` is the plan's real type for the floating-point selectors.
    """
    sel, dt = EXPORTS[what]
    dt = dt or dtype
    if dt is None:
        raise ValueError(f"export {what!r} needs the plan dtype")
    nbytes = lib().fmm_plan_export_size(plan, sel)
    if nbytes < 0:
        raise FmmError(1, f"unknown export {what!r}")
    out = np.empty(nbytes // np.dtype(dt).itemsize, dtype=dt)
    if nbytes:
        _check(lib().fmm_plan_export(plan, sel, out.ctypes.data, nbytes))
    return out


class Plan:
    """RAII wrapper: ``with Plan(n, p, theta, leaf, "f32") as pl: pl.eval(pos, mass, acc, pot)``."""

    def __init__(self, n, p=4, theta=0.7, leaf=32, dtype="f32", f64_ieee=False, m2l_rotation=False, mutual=False):
        self.n, self.p, self.theta, self.leaf = int(n), int(p), float(theta), int(leaf)
        self.dtype = dtype
        self.np_dtype = np.float32 if dtype == "f32" else np.float64
        self.handle = fmm_plan_create(n, p, theta, leaf, FMM_F32 if dtype == "f32" else FMM_F64)
        try:
            if f64_ieee:
                fmm_plan_set_f64_ieee(self.handle, True)
            if m2l_rotation:
                fmm_plan_set_m2l_rotation(self.handle, True)
            if mutual:
                fmm_plan_set_mutual(self.handle, True)
        except FmmError:
            self.close()
            raise

    def eval(self, pos, mass, acc_out, pot_out=None, stream=None):
        fmm_eval(self.handle, pos, mass, acc_out, pot_out, stream)

    def eval_host(self, pos, mass, acc_out, pot_out=None, stream=None):
        fmm_eval_host(self.handle, pos, mass, acc_out, pot_out, stream)

    def kdk_step(self, pos, vel, mass, dt, stream=None):
        fmm_kdk_step(self.handle, pos, vel, mass, dt, stream)

    def kdk_step_lattice(self, pos, vel, mass, dt, pos_exp=-40, vel_exp=-40, stream=None):
        fmm_kdk_step_lattice(self.handle, pos, vel, mass, dt, pos_exp, vel_exp, stream)

    def kdk_reset(self):
        fmm_kdk_reset(self.handle)

    def vjp(self, pos, mass, acc_bar, pot_bar, pos_bar, mass_bar, stream=None):
        fmm_vjp(self.handle, pos, mass, acc_bar, pot_bar, pos_bar, mass_bar, stream)

    def stats(self) -> dict:
        return fmm_plan_stats(self.handle)

    def export(self, what: str) -> np.ndarray:
        return fmm_plan_export(self.handle, what, self.np_dtype)

    def close(self):
        if self.handle:
            fmm_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
