"""Emit ``rotation_gen.cuh``: the rotation-based M2L in real solid harmonics.

jaccpot issue 152 (item 1, "An on-chip-rotation Pallas M2L kernel"): rotate
each source multipole so that the separation lies on the z axis, translate
along z, rotate the local back, with the rotations built on chip from the
separation instead of being read per pair. In the frame where R = |R| z the
translation only couples coefficients of equal order m, which is what makes
the method O(p^3) per pair instead of the O(p^4) of a dense contraction.

Basis. Real regular solid harmonics with Schmidt semi-normalisation and no
Condon-Shortley phase, S_{l,m}(x) for m = -l..l:
    S_{l,0}  = r^l P_l(cos t),
    S_{l,m}  = sqrt(2 (l-m)!/(l+m)!) r^l P_l^m(cos t) cos(m f),
    S_{l,-m} = sqrt(2 (l-m)!/(l+m)!) r^l P_l^m(cos t) sin(m f),   m > 0,
with P_l^m(u) = (1-u^2)^{m/2} d^m P_l/du^m; each is a homogeneous harmonic
polynomial of degree l (expanded exactly with sympy here). All m of one degree
have the same norm, so a rotation acts on each degree by an orthogonal matrix.

Per node (``to_sph``): spherical multipoles Q_{l,m} = sum_j q_j S_{l,m}(s_j),
i.e. Q = A M with A read off the monomial coefficients (times n!) of S_{l,m}.
Per receiver (``from_sph``): the local series sum_{j,m} Ls_{j,m} S_{j,m}(x) as
Cartesian Taylor coefficients, L_k = k! [x^k] of that polynomial.

Per pair (``m2l``), with R = c_A - c_B = |R| (sin t cos f, sin t sin f, cos t):
  1. Q' = W(Rot) Q with Rot = Ry(-t) Rz(-f), so that Rot R = |R| z. A rotation
     about z by a mixes each (m, -m) pair: (q_m, q_-m) ->
     (cos(m a) q_m - sin(m a) q_-m, sin(m a) q_m + cos(m a) q_-m); a rotation
     about y by b is J^T Rz(b) J with J the constant (sparse) matrix of
     Rx(pi/2) per degree. cos(m a), sin(m a) come from the angle's cosine and
     sine by complex multiplication, so no trigonometric call is needed.
  2. The axial translation (the addition theorem for R on the z axis):
        L'_{j,m} = sum_{l <= p-j, l >= |m|} K(j,l,|m|) Q'_{l,m} / |R|^{j+l+1},
        K(j,l,m) = (-1)^{j+m+1} (j+l)! / sqrt((j-m)! (j+m)! (l-m)! (l+m)!),
     with G = 1 and the potential convention Phi = -sum m / r of the other
     operators; the truncation j + l <= p is the total-degree truncation of
     the Cartesian M2L, so the result is the same.
  3. L += W(Rot)^T L' = Rz(f) J^T Rz(t) J L', accumulated per pair.

The generator checks its own tables: the solid harmonics are harmonic and
orthogonal in the sense above, J reproduces Ry(b) = J^T Rz(b) J on random
angles, and A, B invert each other on harmonic polynomials. The host test
compares the generated operators with the oracle's Cartesian M2L for every
order.

Run ``python gen_rotation.py`` to regenerate; the output is committed.
"""
from __future__ import annotations

import math
import os

import numpy as np
import sympy as sp

MAXP = 8
X, Y, Z = sp.symbols("x y z", real=True)


def table(p):
    out = []
    for d in range(p + 1):
        for nx in range(d, -1, -1):
            for ny in range(d - nx, -1, -1):
                out.append((nx, ny, d - nx - ny))
    return out


def cidx(n):
    nx, ny, nz = n
    d = nx + ny + nz
    t = d - nx
    return d * (d + 1) * (d + 2) // 6 + t * (t + 1) // 2 + (t - ny)


def sidx(l, m):
    return l * l + m + l


def solid(l, m):
    """S_{l,m} as an expanded polynomial in x, y, z."""
    u, r = sp.Symbol("u"), sp.Symbol("r", positive=True)
    am = abs(m)
    dP = sp.diff(sp.legendre(l, u), u, am)  # degree l - m, parity l - m
    poly = sp.expand(sp.expand(dP.subs(u, Z / r) * r ** (l - am)).subs(r, sp.sqrt(X * X + Y * Y + Z * Z)))
    w = sp.expand((X + sp.I * Y) ** am)
    part = 1 if m == 0 else (sp.re(w) if m > 0 else sp.im(w))
    norm = 1 if m == 0 else sp.sqrt(2 * sp.Rational(math.factorial(l - am), math.factorial(l + am)))
    return sp.expand(norm * poly * part)


def mono_coeffs(poly, l):
    P = sp.Poly(poly, X, Y, Z)
    return {n: P.coeff_monomial(X ** n[0] * Y ** n[1] * Z ** n[2]) for n in table(l) if sum(n) == l}


def lit(v):
    return f"T({float(v)!r})"


def snap(w):
    """An entry of a real rotation matrix of the harmonics is +-sqrt(rational): round it to that value."""
    from fractions import Fraction
    if w == 0.0:
        return 0.0
    q = Fraction(w * w).limit_denominator(1 << 20)
    exact = math.copysign(float(sp.sqrt(sp.Rational(q.numerator, q.denominator)).evalf(25)), w)
    assert abs(exact - w) < 1e-12, (w, q)
    return exact


def term(c, name):
    """c * name, written without the multiplication for c = +-1."""
    if c == 1.0:
        return name
    if c == -1.0:
        return f"-{name}"
    return f"{lit(c)} * {name}"


class Tables:
    def __init__(self, p):
        self.p = p
        self.S = {(l, m): solid(l, m) for l in range(p + 1) for m in range(-l, l + 1)}
        for (l, m), s in self.S.items():  # harmonic, degree l
            assert sp.expand(sp.diff(s, X, 2) + sp.diff(s, Y, 2) + sp.diff(s, Z, 2)) == 0, (l, m)
        self.C = {k: mono_coeffs(s, k[0]) for k, s in self.S.items()}
        self.J = [self.jmat(l) for l in range(p + 1)]
        self.check_rotation()

    def vec(self, poly, l):
        c = mono_coeffs(poly, l)
        return np.array([float(c[n]) for n in table(l) if sum(n) == l])

    def jmat(self, l):
        """W(J) for J = Rx(pi/2), (x, y, z) -> (x, -z, y): S_l(J s) = W S_l(s)."""
        basis = np.array([self.vec(self.S[(l, m)], l) for m in range(-l, l + 1)]).T
        W = np.zeros((2 * l + 1, 2 * l + 1))
        for m in range(-l, l + 1):
            rotated = sp.expand(self.S[(l, m)].subs({Y: -Z, Z: Y}, simultaneous=True))
            w, res, *_ = np.linalg.lstsq(basis, self.vec(rotated, l), rcond=None)
            assert np.allclose(basis @ w, self.vec(rotated, l), atol=1e-12)
            W[m + l] = w
        W[np.abs(W) < 1e-13] = 0.0
        assert np.allclose(W @ W.T, np.eye(2 * l + 1), atol=1e-12)
        return np.vectorize(snap)(W)

    def check_rotation(self):
        """Ry(b) = J^T Rz(b) J on each degree, checked by evaluating the harmonics at random points."""
        rng = np.random.default_rng(1)
        pts = rng.normal(size=(64, 3))
        b = 0.61
        ry = np.array([[np.cos(b), 0, np.sin(b)], [0, 1, 0], [-np.sin(b), 0, np.cos(b)]])
        for l in range(self.p + 1):
            f = [sp.lambdify((X, Y, Z), self.S[(l, m)], "numpy") for m in range(-l, l + 1)]
            ev = lambda q: np.array([np.broadcast_to(fi(q[:, 0], q[:, 1], q[:, 2]), (len(q),)) for fi in f])
            Wy, *_ = np.linalg.lstsq(ev(pts).T, ev(pts @ ry.T).T, rcond=None)
            Wz = np.eye(2 * l + 1)
            for m in range(1, l + 1):
                c, s = np.cos(m * b), np.sin(m * b)
                Wz[m + l, m + l], Wz[m + l, -m + l], Wz[-m + l, m + l], Wz[-m + l, -m + l] = c, -s, s, c
            assert np.allclose(Wy.T, self.J[l].T @ Wz @ self.J[l], atol=1e-10), l

    def K(self, j, l, m):
        return (-1) ** (j + m + 1) * math.factorial(j + l) / math.sqrt(
            math.factorial(j - m) * math.factorial(j + m) * math.factorial(l - m) * math.factorial(l + m))


def zrot(arr, p, c, s, sign, degrees):
    """Lines rotating arr about z: (a_m, a_-m) -> (c_m a_m - sign s_m a_-m, sign s_m a_m + c_m a_-m)."""
    b = []
    for l in degrees:
        for m in range(1, l + 1):
            i, k = sidx(l, m), sidx(l, -m)
            sp_, sn = ("-", "+") if sign > 0 else ("+", "-")
            b.append(f"  {{ const T u = {arr}[{i}], v = {arr}[{k}]; "
                     f"{arr}[{i}] = c{c}{m} * u {sp_} s{c}{m} * v; {arr}[{k}] = c{c}{m} * v {sn} s{c}{m} * u; }}")
    return b


def jmul(T, src, dst, degrees, transpose):
    """dst = W(J) src (or its transpose), only the nonzero entries."""
    b = []
    for l in degrees:
        W = T.J[l].T if transpose else T.J[l]
        for mo in range(-l, l + 1):
            terms = []
            for mi in range(-l, l + 1):
                w = W[mo + l, mi + l]
                if w == 0.0:
                    continue
                terms.append(term(w, f"{src}[{sidx(l, mi)}]"))
            b.append(f"  {dst}[{sidx(l, mo)}] = " + (" + ".join(terms) if terms else "T(0)") + ";")
    return b


def gen_struct(p):
    T = Tables(p)
    ns = (p + 1) ** 2
    nc = len(table(p))
    out = [f"template <> struct Rot<{p}> {{", f"  static constexpr int NS = {ns};"]
    # to_sph: Q = A M
    b = ["template <class T> static __device__ __forceinline__ void to_sph(const T* M, T* Q) {"]
    for l in range(p + 1):
        for m in range(-l, l + 1):
            terms = []
            for n, a in T.C[(l, m)].items():
                if a == 0:
                    continue
                f = math.factorial(n[0]) * math.factorial(n[1]) * math.factorial(n[2])
                terms.append(term(float(a) * f, f"M[{cidx(n)}]"))
            b.append(f"  Q[{sidx(l, m)}] = " + (" + ".join(terms) if terms else "T(0)") + ";")
    b.append("}")
    # from_sph: L_k = k! [x^k] sum_m Ls_m S_m
    b.append("template <class T> static __device__ __forceinline__ void from_sph(const T* Ls, T* L) {")
    for n in table(p):
        l = sum(n)
        f = math.factorial(n[0]) * math.factorial(n[1]) * math.factorial(n[2])
        terms = []
        for m in range(-l, l + 1):
            a = T.C[(l, m)][n]
            if a != 0:
                terms.append(term(float(a) * f, f"Ls[{sidx(l, m)}]"))
        b.append(f"  L[{cidx(n)}] = " + (" + ".join(terms) if terms else "T(0)") + ";")
    b.append("}")
    # the pair operator
    b.append("template <class T> static __device__ __forceinline__ void m2l(const T* Q, T rx, T ry, T rz, T* Ls) {")
    b.append("  const T rho2 = rx * rx + ry * ry;")
    b.append("  const T r2 = rho2 + rz * rz;")
    b.append("  const T ir = rsqrt_t(r2);")
    if p == 0:
        b.append("  Ls[0] -= Q[0] * ir;")
        b.append("}")
        out += ["  " + l for l in b]
        out.append("};")
        return out
    b.append("  const T irho = rho2 > T(0) ? rsqrt_t(rho2) : T(0);")
    b.append("  // the azimuth f and polar angle t of R (any azimuth on the z axis)")
    b.append("  const T cf1 = rho2 > T(0) ? rx * irho : T(1), sf1 = ry * irho;")
    b.append("  const T ct1 = rz * ir, st1 = rho2 * irho * ir;")
    for a in ("f", "t"):
        for m in range(2, p + 1):
            b.append(f"  const T c{a}{m} = c{a}{m - 1} * c{a}1 - s{a}{m - 1} * s{a}1, "
                     f"s{a}{m} = s{a}{m - 1} * c{a}1 + c{a}{m - 1} * s{a}1;")
    b.append("  T ip[%d];" % (p + 2))
    b.append("  ip[0] = T(1);")
    for k in range(1, p + 2):
        b.append(f"  ip[{k}] = ip[{k - 1}] * ir;")
    b.append(f"  T q[{ns}], w[{ns}];")
    b.append(f"  for (int i = 0; i < {ns}; ++i) q[i] = Q[i];")
    allg = list(range(p + 1))
    b.append("  // Q' = J^T Rz(-t) J Rz(-f) Q")
    b += zrot("q", p, "f", None, -1, allg)
    b += jmul(T, "q", "w", allg, False)
    b += zrot("w", p, "t", None, -1, allg)
    b += jmul(T, "w", "q", allg, True)
    b.append("  // the translation along z, each degree scaled by its power of 1/|R|")
    for l in allg:
        for m in range(-l, l + 1):
            b.append(f"  q[{sidx(l, m)}] *= ip[{l}];")
    for j in allg:
        for m in range(-j, j + 1):
            terms = []
            for l in range(abs(m), p - j + 1):
                terms.append(term(T.K(j, l, abs(m)), f"q[{sidx(l, m)}]"))
            b.append(f"  w[{sidx(j, m)}] = (" + " + ".join(terms) + f") * ip[{j + 1}];" if terms
                     else f"  w[{sidx(j, m)}] = T(0);")
    b.append("  // L += Rz(f) J^T Rz(t) J L'")
    b += jmul(T, "w", "q", allg, False)
    b += zrot("q", p, "t", None, +1, allg)
    b += jmul(T, "q", "w", allg, True)
    b += zrot("w", p, "f", None, +1, allg)
    b.append(f"  for (int i = 0; i < {ns}; ++i) Ls[i] += w[i];")
    b.append("}")
    out += ["  " + l for l in b]
    out.append("};")
    return out


def main():
    out = ["// Generated by gen_rotation.py -- do not edit by hand.",
           "// Rotation-based M2L in real solid harmonics for orders 0..8 (see the generator's docstring).",
           "#pragma once",
           "",
           '#include "expansions_gen.cuh"',
           "",
           "namespace bfm {",
           "",
           "template <int P> struct Rot;",
           ""]
    for p in range(MAXP + 1):
        out += gen_struct(p)
        out.append("")
    out.append("}  // namespace bfm")
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rotation_gen.cuh")
    with open(path, "w") as f:
        f.write("\n".join(out) + "\n")
    print(path, len(out), "lines")


if __name__ == "__main__":
    main()
