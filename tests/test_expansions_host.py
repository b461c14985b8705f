"""The CUDA path's generated expansion operators, compiled for the host,
against the oracle's operators (independent code) for every order 0..8.

This checks the code generator on the CPU; the GPU parity tests check the
same operators as they run inside the kernels."""
import ctypes as C
import os
import subprocess

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "shim", "expansions_host.cpp")
GEN = os.path.join(HERE, "..", "body_forces_morton_b300", "csrc", "expansions_gen.cuh")


@pytest.fixture(scope="module")
def shim(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("shim") / "libexpshim.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-ffp-contract=off", "-shared", "-fPIC", "-o", out, SRC],
                   check=True)
    lib = C.CDLL(out)
    for f in ("shim_op_f64", "shim_op_f32"):
        getattr(lib, f).argtypes = [C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
        getattr(lib, f).restype = C.c_int
    return lib


def call(lib, p, op, a, v, nout, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    v = np.ascontiguousarray(v, dtype=dtype)
    out = np.zeros(nout, dtype=dtype)
    f = lib.shim_op_f64 if dtype == np.float64 else lib.shim_op_f32
    assert f(p, op, a.ctypes.data, v.ctypes.data, out.ctypes.data) == 0
    return out.astype(np.float64)


@pytest.mark.parametrize("p", range(9))
@pytest.mark.parametrize("dtype,rtol", [(np.float64, 1e-12), (np.float32, 2e-4)])
def test_generated_operators_match_oracle(shim, p, dtype, rtol):
    rng = np.random.default_rng(100 + p)
    nc = oracle.ncoef(p)
    # P2M: one particle
    s, m = rng.normal(size=3) * 0.1, 0.7
    got = call(shim, p, 0, np.zeros(1), [*s, m], nc, dtype)
    want = oracle.p2m(p, s[None, :], [m], np.zeros(3))
    np.testing.assert_allclose(got, want, rtol=rtol, atol=rtol * np.abs(want).max())
    # M2M, M2L, L2L on random coefficient vectors
    M = rng.normal(size=nc)
    d = rng.normal(size=3) * 0.2
    R = np.array([1.1, -0.6, 0.8])
    for op, fn, arg in ((1, oracle.m2m, d), (2, oracle.m2l, R), (3, oracle.l2l, d)):
        got = call(shim, p, op, M, arg, nc, dtype)
        want = fn(p, M, arg)
        np.testing.assert_allclose(got, want, rtol=rtol, atol=rtol * np.abs(want).max(), err_msg=f"op {op}")
    # reduced (trace-free) M2L: reduce the moments, contract, expand the locals
    got = call(shim, p, 5, M, R, nc, dtype)
    want = oracle.m2l(p, M, R)
    np.testing.assert_allclose(got, want, rtol=rtol, atol=rtol * np.abs(want).max(), err_msg="reduced m2l")
    # both directions of one pair from one derivative tensor (mutual M2L): L_A from M_B at R and
    # L_B from M_A at -R, each against the oracle's one-directional M2L
    MA = rng.normal(size=nc)
    got = call(shim, p, 6, np.concatenate([MA, M]), R, 2 * nc, dtype)
    for half, want in ((got[:nc], oracle.m2l(p, M, R)), (got[nc:], oracle.m2l(p, MA, -R))):
        np.testing.assert_allclose(half, want, rtol=rtol, atol=rtol * np.abs(want).max(), err_msg="pair m2l")
    # rotation-based M2L (rotate R onto z, translate along z, rotate back) against the Cartesian M2L,
    # for a general separation and for separations on the +z and -z axes (azimuth undefined)
    for Rr in (R, np.array([0.0, 0.0, 1.7]), np.array([0.0, 0.0, -0.9]), np.array([-0.3, 0.0, 0.0])):
        got = call(shim, p, 9, M, Rr, nc, dtype)
        want = oracle.m2l(p, M, Rr)
        np.testing.assert_allclose(got, want, rtol=rtol, atol=rtol * np.abs(want).max(), err_msg=f"rotation m2l {Rr}")
    # the VJP's operators: a source with monopole q and dipole d, and the local series' Hessian
    q, dd = 0.4, rng.normal(size=3)
    got = call(shim, p, 7, np.zeros(1), [*s, q, *dd], nc, dtype)
    want = oracle.p2m_dipole(p, s[None, :], [q], dd[None, :], np.zeros(3))
    np.testing.assert_allclose(got, want, rtol=rtol, atol=rtol * np.abs(want).max(), err_msg="p2m_dip")
    dxh = rng.normal(size=3) * 0.1
    got = call(shim, p, 8, M, dxh, 6, dtype)
    want = oracle.l2p_hess(p, M, dxh)
    np.testing.assert_allclose(got, want, rtol=rtol, atol=rtol * max(np.abs(want).max(), 1e-300),
                               err_msg="l2p_hess")
    # L2P
    dx = rng.normal(size=3) * 0.1
    got = call(shim, p, 4, M, dx, 4, dtype)
    phi, acc = oracle.l2p(p, M, dx)
    want = np.array([phi, *acc])
    np.testing.assert_allclose(got, want, rtol=rtol, atol=rtol * np.abs(want).max())
