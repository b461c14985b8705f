"""Emit ``expansions_gen.cuh``: fully unrolled Cartesian expansion operators.

For every order P in 0..8 this writes a specialisation ``Exp<P>`` with device
functions templated on the real type (float / double):

  p2m  M_n  += m s^n / n!                                  (JZ-FMM moment eqs.)
  m2m  Mp_n += sum_{k<=n} Mc_k d^{n-k} / (n-k)!              (upward translation)
  m2l  L_k  += -sum_{|n|<=P-|k|} (-1)^{|n|} M_n D^{n+k}(R)   (M2L eqs.), with
       D^n = d^n(1/r) from the recurrence
       l r^2 D^n = -(2l-1) sum_i n_i R_i D^{n-e_i} - (l-1) sum_i n_i(n_i-1) D^{n-2e_i}
  l2l  Lc_k += sum_{j>=k} Lp_j e^{j-k} / (j-k)!               (downward translation)
  l2p  phi = sum_k L_k x^k/k!,  a = -sum_k L_{k+e_a} x^k/k!   (Taylor eq.)
  p2m_dip   M_n += q s^n/n! + sum_a d_a s^{n-e_a}/(n-e_a)!     (sources of the
            FMM VJP: monopole q and dipole d; JZ-FMM page, "Differentiating
            the force calculation")
  l2p_hess  H_ab += sum_{|k|<=P-2} L_{k+e_a+e_b} x^k/k!        (the next higher
            derivative of the local series, for the same VJP)

Every index is a compile-time constant, so the coefficient arrays of the
callers live in registers. Coefficient order: graded by total degree; within
a degree the x exponent descends, then the y exponent.

Reduced (trace-free) M2L. D^m is harmonic, so D^m = -(D^{m-2e_z+2e_x} +
D^{m-2e_z+2e_y}) whenever m_z >= 2. Applied to the contraction, M_n with
n_z >= 2 folds into "reduced" moments indexed by n_z <= 1 (2l+1 per degree l),
and the locals L_k with k_z >= 2 follow from those with k_z <= 1 by the same
identity (their truncated sums obey it term by term). ``m2l_r`` contracts
reduced moments into reduced locals ((p+1)^2 each; 155 instead of 210 terms at
p = 4) and needs D^m only for m_z <= 2, the m_z = 2 ones from the identity;
``reduce_m`` and ``expand_l`` convert from and to the full coefficients.
``m2l_r_pair`` is both directions of one pair from one derivative tensor (for
a mutual FMM): D^m(-R) = (-1)^{|m|} D^m(R) gives the reverse contraction.

It also writes ``expansions_df_gen.cuh``: ``ExpDF<P>::m2l_r`` for P <= 4, the
reduced M2L with every value a double-float (dfloat.cuh): the derivative
recurrence in double-word operations (constants split into fp32 pairs at
generation time, exact ones applied with the cheaper forms), the contraction
as lazily normalised product accumulations.

Run ``python gen_expansions.py`` to regenerate; the output is committed.
"""
from __future__ import annotations

import os
from math import factorial

MAXP = 8


def ncoef(p):
    return (p + 1) * (p + 2) * (p + 3) // 6


def idx(n):
    nx, ny, nz = n
    d = nx + ny + nz
    t = d - nx
    return d * (d + 1) * (d + 2) // 6 + t * (t + 1) // 2 + (t - ny)


def table(p):
    out = []
    for d in range(p + 1):
        for nx in range(d, -1, -1):
            for ny in range(d - nx, -1, -1):
                out.append((nx, ny, d - nx - ny))
    assert [idx(n) for n in out] == list(range(len(out)))
    return out


def lit(v):
    """A real literal converted to T at compile time."""
    return f"T({float(v)!r})"


AX = "xyz"


def mono_recurrence(p, src, var, name, first=None):
    """Lines computing name[n] = (first) * var^n / n! for |n| <= p.

    ``var`` is a prefix: the scaled coordinates var{axis}{k} = var_axis / k
    must be defined by the caller for k = 1..p.
    """
    lines = []
    mi = table(p)
    lines.append(f"T {name}[{len(mi)}];")
    lines.append(f"{name}[0] = {first if first else 'T(1)'};")
    for n in mi[1:]:
        i = 0 if n[0] > 0 else (1 if n[1] > 0 else 2)
        m = list(n)
        m[i] -= 1
        lines.append(f"{name}[{idx(n)}] = {name}[{idx(tuple(m))}] * {var}{AX[i]}{n[i]};")
    return lines


def scaled_coords(p, var, x, y, z):
    lines = []
    if p == 0:
        return lines
    for a, c in zip(AX, (x, y, z)):
        lines.append(f"const T {var}{a}1 = {c};")
        for k in range(2, p + 1):
            lines.append(f"const T {var}{a}{k} = {c} * {lit(1.0 / k)};")
    return lines


def gen_p2m(p):
    b = ["template <class T> static __device__ __forceinline__ void p2m(T sx, T sy, T sz, T m, T* M) {"]
    if p == 0:
        b.append("  (void)sx; (void)sy; (void)sz;")
    b += ["  " + l for l in scaled_coords(p, "s", "sx", "sy", "sz")]
    b += ["  " + l for l in mono_recurrence(p, None, "s", "t", first="m")]
    for n in table(p):
        b.append(f"  M[{idx(n)}] += t[{idx(n)}];")
    b.append("}")
    return b


def gen_m2m(p):
    b = ["template <class T> static __device__ __forceinline__ void m2m(const T* Mc, T dx, T dy, T dz, T* Mp) {"]
    if p == 0:
        b.append("  (void)dx; (void)dy; (void)dz;")
    if p > 0:
        b += ["  " + l for l in scaled_coords(p, "d", "dx", "dy", "dz")]
        b += ["  " + l for l in mono_recurrence(p, None, "d", "u")]
    for n in table(p):
        terms = []
        for k in table(p):
            if k[0] <= n[0] and k[1] <= n[1] and k[2] <= n[2]:
                q = (n[0] - k[0], n[1] - k[1], n[2] - k[2])
                if q == (0, 0, 0):
                    terms.append(f"Mc[{idx(k)}]")
                else:
                    terms.append(f"Mc[{idx(k)}] * u[{idx(q)}]")
        b.append(f"  Mp[{idx(n)}] += " + " + ".join(terms) + ";")
    b.append("}")
    return b


def gen_derivs(p):
    """Lines building D[ncoef(p)] from rx, ry, rz (1/r derivative tensor)."""
    mi = table(p)
    L = [f"T D[{len(mi)}];",
         "const T r2 = rx * rx + ry * ry + rz * rz;",
         "D[0] = rsqrt_t(r2);"]
    if p == 0:
        return L
    L.append("const T ir2 = D[0] * D[0];")
    L.append("const T ax = rx * ir2, ay = ry * ir2, az = rz * ir2;")
    for a in AX:
        for k in range(2, p + 1):
            L.append(f"const T a{a}{k} = a{a} * {lit(k)};")
    for l in range(2, p + 1):
        L.append(f"const T c2_{l} = ir2 * {lit(-(l - 1) / l)};")
    for n in mi[1:]:
        l = sum(n)
        s1 = []
        s2 = []
        for i in range(3):
            if n[i] >= 1:
                m = list(n)
                m[i] -= 1
                coef = f"a{AX[i]}" if n[i] == 1 else f"a{AX[i]}{n[i]}"
                s1.append(f"{coef} * D[{idx(tuple(m))}]")
            if n[i] >= 2:
                m = list(n)
                m[i] -= 2
                s2.append(f"{lit(n[i] * (n[i] - 1))} * D[{idx(tuple(m))}]")
        c1 = lit(-(2 * l - 1) / l)
        expr = f"{c1} * ({' + '.join(s1)})"
        if s2:
            expr += f" + c2_{l} * ({' + '.join(s2)})"
        L.append(f"D[{idx(n)}] = {expr};")
    return L


def gen_m2l(p):
    b = ["template <class T> static __device__ __forceinline__ void m2l(const T* M, T rx, T ry, T rz, T* L) {"]
    b += ["  " + l for l in gen_derivs(p)]
    mi = table(p)
    for k in mi:
        lk = sum(k)
        for n in mi:
            ln = sum(n)
            if ln + lk > p:
                continue
            j = idx((n[0] + k[0], n[1] + k[1], n[2] + k[2]))
            op = "+=" if ln % 2 == 1 else "-="
            b.append(f"  L[{idx(k)}] {op} M[{idx(n)}] * D[{j}];")
    b.append("}")
    return b


def reduced_table(p):
    """Multi-indices with n_z <= 1 in coefficient order, and their reduced index."""
    out = [n for n in table(p) if n[2] <= 1]
    return out, {n: i for i, n in enumerate(out)}


def reduction(n, rmap):
    """n as a combination of reduced indices, by the trace identity: {ridx: coef}."""
    if n[2] <= 1:
        return {rmap[n]: 1}
    res = {}
    for m in ((n[0] + 2, n[1], n[2] - 2), (n[0], n[1] + 2, n[2] - 2)):
        for k, c in reduction(m, rmap).items():
            res[k] = res.get(k, 0) - c
    return res


def lin_comb(terms):
    """'a + b - 2 * c' from [(coef, expr)]."""
    out = ""
    for c, e in terms:
        if c == 0:
            continue
        mag = abs(c)
        t = e if mag == 1 else f"{lit(mag)} * {e}"
        if not out:
            out = t if c > 0 else f"-({t})"
        else:
            out += f" + {t}" if c > 0 else f" - {t}"
    return out or "T(0)"


def gen_reduce_m(p):
    red, rmap = reduced_table(p)
    acc = {i: [] for i in range(len(red))}
    for n in table(p):
        for r, c in reduction(n, rmap).items():
            acc[r].append((c, f"M[{idx(n)}]"))
    b = ["template <class T> static __device__ __forceinline__ void reduce_m(const T* M, T* Mr) {"]
    for r in range(len(red)):
        b.append(f"  Mr[{r}] = {lin_comb(acc[r])};")
    b.append("}")
    return b


def gen_expand_l(p):
    red, rmap = reduced_table(p)
    b = ["template <class T> static __device__ __forceinline__ void expand_l(const T* Lr, T* L) {"]
    for k in table(p):
        terms = sorted(reduction(k, rmap).items())
        b.append(f"  L[{idx(k)}] = {lin_comb([(c, f'Lr[{r}]') for r, c in terms])};")
    b.append("}")
    return b


def reduced_derivs(p):
    """(slot map, lines) building D^m for m_z <= 2, |m| <= p, in a compact array."""
    mi = [m for m in table(p) if m[2] <= 2]
    slot = {m: i for i, m in enumerate(mi)}
    return mi, slot


def gen_m2l_r(p):
    red, rmap = reduced_table(p)
    b = ["template <class T> static __device__ __forceinline__ void m2l_r(const T* M, T rx, T ry, T rz, T* L) {"]
    b += reduced_derivs_body(p)
    b += reduced_contraction(p, "M", "L", 0)
    b.append("}")
    return b


def gen_m2l_r_pair(p):
    """Both directions of one M2L pair from one derivative tensor (mutual FMM):
    LA from MB with R = c_A - c_B as in m2l_r, and LB from MA with -R, using
    D^m(-R) = (-1)^{|m|} D^m(R): LB_k += -(-1)^{|k|} sum_n MA_n D^{n+k}(R)."""
    b = ["template <class T> static __device__ __forceinline__ void m2l_r_pair(const T* MA, const T* MB, T rx, T ry, "
         "T rz, T* LA, T* LB) {"]
    b += reduced_derivs_body(p)
    b += reduced_contraction(p, "MB", "LA", 0)
    b += reduced_contraction(p, "MA", "LB", 1)
    b.append("}")
    return b


def reduced_contraction(p, m_name, l_name, mirrored):
    """Contraction lines L_k += -sum (-1)^{|n|} M_n D^{n+k}; mirrored: the sign (-1)^{|k|} instead."""
    red, rmap = reduced_table(p)
    mi, slot = reduced_derivs(p)
    b = []
    for k in red:
        for n in red:
            if sum(n) + sum(k) > p:
                continue
            m = (n[0] + k[0], n[1] + k[1], n[2] + k[2])
            odd = (sum(k) if mirrored else sum(n)) % 2 == 1
            op = "+=" if odd else "-="
            b.append(f"  {l_name}[{rmap[k]}] {op} {m_name}[{rmap[n]}] * D[{slot[m]}];")
    return b


def reduced_derivs_body(p):
    """Lines building D[] (the reduced derivative tensor of 1/r at (rx, ry, rz)).

    The recurrence l r^2 D^n = -(2l-1) sum_i n_i R_i D^{n-e_i}
    - (l-1) sum_i n_i (n_i-1) D^{n-2e_i} with its constants folded into
    per-level coefficients, A_{l,i,m} = a_i (-(2l-1)/l) m (a = R / r^2) and
    C_{l,c} = (1/r^2) (-(l-1)/l) c, so each D^n is a sum of coefficient-times-D
    terms (one product and a chain of fused multiply-adds)."""
    mi, slot = reduced_derivs(p)
    b = [f"  T D[{len(mi)}];",
         "  const T r2 = rx * rx + ry * ry + rz * rz;",
         f"  D[{slot[(0, 0, 0)]}] = rsqrt_t(r2);"]
    if p > 0:
        b.append("  const T ir2 = D[0] * D[0];")
        b.append("  const T ax = rx * ir2, ay = ry * ir2, az = rz * ir2;")
    need_a, need_c, terms_of = [], [], {}
    for n in mi[1:]:
        if n[2] == 2:
            continue
        l = sum(n)
        terms = []
        for i in range(3):
            if n[i] >= 1:
                m = list(n)
                m[i] -= 1
                if l == 1:
                    terms.append((f"(-a{AX[i]})", slot[tuple(m)]))
                else:
                    key = (l, i, n[i])
                    if key not in need_a:
                        need_a.append(key)
                    terms.append((f"A{l}{AX[i]}{n[i]}", slot[tuple(m)]))
            if n[i] >= 2:
                m = list(n)
                m[i] -= 2
                key = (l, n[i] * (n[i] - 1))
                if key not in need_c:
                    need_c.append(key)
                terms.append((f"C{l}_{key[1]}", slot[tuple(m)]))
        terms_of[n] = terms
    for l, i, m in need_a:
        b.append(f"  const T A{l}{AX[i]}{m} = a{AX[i]} * {lit(-(2 * l - 1) / l * m)};")
    for l, c in need_c:
        b.append(f"  const T C{l}_{c} = ir2 * {lit(-(l - 1) / l * c)};")
    for n in mi[1:]:
        if n[2] == 2:
            continue
        b.append(f"  D[{slot[n]}] = " + " + ".join(f"{c} * D[{sl}]" for c, sl in terms_of[n]) + ";")
    for n in mi:
        if n[2] == 2:
            a_, b_ = (n[0] + 2, n[1], 0), (n[0], n[1] + 2, 0)
            b.append(f"  D[{slot[n]}] = -(D[{slot[a_]}] + D[{slot[b_]}]);")
    return b


def gen_l2l(p):
    b = ["template <class T> static __device__ __forceinline__ void l2l(const T* Lp, T ex, T ey, T ez, T* Lc) {"]
    if p == 0:
        b.append("  (void)ex; (void)ey; (void)ez;")
    if p > 0:
        b += ["  " + l for l in scaled_coords(p, "e", "ex", "ey", "ez")]
        b += ["  " + l for l in mono_recurrence(p, None, "e", "u")]
    mi = table(p)
    for k in mi:
        terms = []
        for j in mi:
            if j[0] >= k[0] and j[1] >= k[1] and j[2] >= k[2]:
                q = (j[0] - k[0], j[1] - k[1], j[2] - k[2])
                terms.append(f"Lp[{idx(j)}]" if q == (0, 0, 0) else f"Lp[{idx(j)}] * u[{idx(q)}]")
        b.append(f"  Lc[{idx(k)}] += " + " + ".join(terms) + ";")
    b.append("}")
    return b


def gen_l2p(p):
    b = ["template <class T> static __device__ __forceinline__ void l2p(const T* L, T dx, T dy, T dz,",
         "                                                        T& phi, T& ax, T& ay, T& az) {"]
    if p > 0:
        b += ["  " + l for l in scaled_coords(p, "x", "dx", "dy", "dz")]
        b += ["  " + l for l in mono_recurrence(p, None, "x", "u")]
    else:
        b.append("  (void)dx; (void)dy; (void)dz;")
        b.append("  T u[1]; u[0] = T(1);")
    mi = table(p)
    b.append("  T f = T(0), gx = T(0), gy = T(0), gz = T(0);")
    for k in mi:
        b.append(f"  f += L[{idx(k)}] * u[{idx(k)}];")
        if sum(k) < p:
            for a, g in zip(range(3), ("gx", "gy", "gz")):
                q = list(k)
                q[a] += 1
                b.append(f"  {g} += L[{idx(tuple(q))}] * u[{idx(k)}];")
    b.append("  phi += f; ax -= gx; ay -= gy; az -= gz;")
    b.append("}")
    return b


def gen_p2m_dip(p):
    """Moments of one source with monopole q and dipole (dx, dy, dz) at offset s:
    M_n += q s^n / n! + sum_a d_a s^{n - e_a} / (n - e_a)! (the FMM VJP's sources)."""
    b = ["template <class T> static __device__ __forceinline__ void p2m_dip(T sx, T sy, T sz, T q, T dx, T dy, T dz,"
         " T* M) {"]
    if p == 0:
        b.append("  (void)sx; (void)sy; (void)sz; (void)dx; (void)dy; (void)dz;")
    b += ["  " + l for l in scaled_coords(p, "s", "sx", "sy", "sz")]
    b += ["  " + l for l in mono_recurrence(p, None, "s", "t")]
    for n in table(p):
        terms = [f"q * t[{idx(n)}]"]
        for a, d in zip(range(3), ("dx", "dy", "dz")):
            if n[a] >= 1:
                m = list(n)
                m[a] -= 1
                terms.append(f"{d} * t[{idx(tuple(m))}]")
        b.append(f"  M[{idx(n)}] += " + " + ".join(terms) + ";")
    b.append("}")
    return b


def gen_l2p_hess(p):
    """Hessian (xx, xy, xz, yy, yz, zz) of the local series at offset (dx, dy, dz), added to H:
    d_a d_b Phi = sum_{|k| <= p - 2} L_{k + e_a + e_b} dx^k / k!."""
    b = ["template <class T> static __device__ __forceinline__ void l2p_hess(const T* L, T dx, T dy, T dz, T* H) {"]
    if p < 2:
        b.append("  (void)L; (void)dx; (void)dy; (void)dz; (void)H;")
        b.append("}")
        return b
    q = p - 2
    if q > 0:
        b += ["  " + l for l in scaled_coords(q, "x", "dx", "dy", "dz")]
        b += ["  " + l for l in mono_recurrence(q, None, "x", "u")]
    else:
        b.append("  (void)dx; (void)dy; (void)dz;")
        b.append("  T u[1]; u[0] = T(1);")
    pairs = [(0, 0), (0, 1), (0, 2), (1, 1), (1, 2), (2, 2)]
    for h, (a1, a2) in enumerate(pairs):
        terms = []
        for k in table(q):
            m = list(k)
            m[a1] += 1
            m[a2] += 1
            terms.append(f"L[{idx(tuple(m))}] * u[{idx(k)}]")
        b.append(f"  H[{h}] += " + " + ".join(terms) + ";")
    b.append("}")
    return b


MAXP_DF = 4


def _f32(c):
    import struct
    return struct.unpack("f", struct.pack("f", c))[0]


def df_cmul(x, c):
    """Double-float x times the real constant c."""
    from math import frexp
    if c == 1:
        return x
    if c == -1:
        return f"df_neg({x})"
    if frexp(abs(c))[0] == 0.5:
        return f"df_scale({x}, {c!r}f)"
    if _f32(c) == c:
        return f"df_mulf({x}, {c!r}f)"
    h = _f32(c)
    lo = _f32(c - h)
    return f"df_mul({x}, df_make({h!r}f, {lo!r}f))"


def df_sum(terms):
    acc = terms[0]
    for t in terms[1:]:
        acc = f"df_add({acc}, {t})"
    return acc


def gen_m2l_df(p):
    """Double-float reduced M2L: m2l_r with double-word operations and product accumulation."""
    red, rmap = reduced_table(p)
    mi, slot = reduced_derivs(p)
    b = ["static __device__ __forceinline__ void m2l_r(const df* M, df rx, df ry, df rz, dacc* L) {",
         f"  df D[{len(mi)}];",
         "  const df r2 = df_add(df_add(df_sqr(rx), df_sqr(ry)), df_sqr(rz));",
         f"  D[{slot[(0, 0, 0)]}] = df_rsqrt(r2);"]
    if p > 0:
        b.append("  const df ir2 = df_sqr(D[0]);")
        b.append("  const df ax = df_mul(rx, ir2), ay = df_mul(ry, ir2), az = df_mul(rz, ir2);")
        for a in AX:
            for k in range(2, p + 1):
                b.append(f"  const df a{a}{k} = {df_cmul('a' + a, float(k))};")
        for l in range(2, p + 1):
            b.append(f"  const df c2_{l} = {df_cmul('ir2', -(l - 1) / l)};")
    for n in mi[1:]:
        if n[2] == 2:
            continue
        l = sum(n)
        s1, s2 = [], []
        for i in range(3):
            if n[i] >= 1:
                m = list(n)
                m[i] -= 1
                coef = f"a{AX[i]}" if n[i] == 1 else f"a{AX[i]}{n[i]}"
                s1.append(f"df_mul({coef}, D[{slot[tuple(m)]}])")
            if n[i] >= 2:
                m = list(n)
                m[i] -= 2
                s2.append(df_cmul(f"D[{slot[tuple(m)]}]", float(n[i] * (n[i] - 1))))
        expr = df_cmul(df_sum(s1), -(2 * l - 1) / l)
        if s2:
            expr = f"df_add({expr}, df_mul(c2_{l}, {df_sum(s2)}))"
        b.append(f"  D[{slot[n]}] = {expr};")
    for n in mi:
        if n[2] == 2:
            a_, b_ = (n[0] + 2, n[1], 0), (n[0], n[1] + 2, 0)
            b.append(f"  D[{slot[n]}] = df_neg(df_add(D[{slot[a_]}], D[{slot[b_]}]));")
    for k in red:
        for n in red:
            if sum(n) + sum(k) > p:
                continue
            m = (n[0] + k[0], n[1] + k[1], n[2] + k[2])
            mn = f"M[{rmap[n]}]" if sum(n) % 2 == 1 else f"df_neg(M[{rmap[n]}])"
            b.append(f"  mac(L[{rmap[k]}], {mn}, D[{slot[m]}]);")
    b.append("}")
    return b


def main_df():
    out = ["// Generated by gen_expansions.py -- do not edit by hand.",
           "// Double-float M2L for orders 0..4 (see the generator's docstring).",
           "#pragma once",
           "",
           '#include "dfloat.cuh"',
           "",
           "namespace bfm {",
           "",
           "template <int P> struct ExpDF;",
           ""]
    for p in range(MAXP_DF + 1):
        out.append(f"template <> struct ExpDF<{p}> {{")
        out.append(f"  static constexpr int NC = {ncoef(p)};")
        out.append(f"  static constexpr int NRC = {(p + 1) ** 2};")
        out += ["  " + l for l in gen_m2l_df(p)]
        out.append("};")
        out.append("")
    out.append("}  // namespace bfm")
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "expansions_df_gen.cuh")
    with open(path, "w") as f:
        f.write("\n".join(out) + "\n")
    print(path, len(out), "lines")


def main():
    out = ["// Generated by gen_expansions.py -- do not edit by hand.",
           "// Unrolled Cartesian expansion operators for orders 0..8 (see the generator's docstring).",
           "#pragma once",
           "",
           "namespace bfm {",
           "",
           "#ifndef BFM_HOST_SHIM",
           "__device__ __forceinline__ float rsqrt_t(float x) { return rsqrtf(x); }",
           "__device__ __forceinline__ double rsqrt_t(double x) { return rsqrt(x); }",
           "#endif",
           "",
           "template <int P> struct Exp;",
           ""]
    for p in range(MAXP + 1):
        out.append(f"template <> struct Exp<{p}> {{")
        out.append(f"  static constexpr int NC = {ncoef(p)};")
        out.append(f"  static constexpr int NRC = {(p + 1) ** 2};  // reduced (n_z <= 1) coefficients")
        for gen in (gen_p2m, gen_m2m, gen_m2l, gen_l2l, gen_l2p, gen_reduce_m, gen_expand_l, gen_m2l_r,
                    gen_m2l_r_pair, gen_p2m_dip, gen_l2p_hess):
            out += ["  " + l for l in gen(p)]
        out.append("};")
        out.append("")
    out.append("}  // namespace bfm")
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "expansions_gen.cuh")
    with open(path, "w") as f:
        f.write("\n".join(out) + "\n")
    print(path, sum(1 for _ in out), "lines")
    main_df()


if __name__ == "__main__":
    main()
