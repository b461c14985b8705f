// Double-float ("double-word") arithmetic on the FP32 pipe for fp64 plans.
//
// A value is an unevaluated sum h + l of two fp32 numbers with |l| <= ulp(h)/2,
// about 48 significant bits. Building blocks are the error-free
// transformations of Dekker and Knuth (two_sum, fast_two_sum, and two_prod via
// FMA) and the double-word algorithms of Joldes, Muller and Popescu ("Tight and
// rigorous error bounds for basic building blocks of double-word arithmetic",
// ACM TOMS 2017): the "sloppy" addition, whose error is ~2^-47 of |x| + |y|,
// and the FMA-based multiplication. Every operation is written with the
// round-to-nearest intrinsics so the compiler cannot contract or reassociate
// the sums whose rounding errors are being captured.
#pragma once

#include "common.cuh"

namespace bfm {

struct __align__(8) df {
    float h, l;
    df() = default;
    __host__ __device__ constexpr df(float h_, float l_) : h(h_), l(l_) {}
    // from a constant of the generated expansion code (split at compile time for literals)
    __host__ __device__ constexpr df(double v) : h((float)v), l((float)(v - (double)(float)v)) {}
};

__device__ __forceinline__ df df_make(float h, float l)
{
    df r;
    r.h = h;
    r.l = l;
    return r;
}

__device__ __forceinline__ df df_from(double v)
{
    df r;
    r.h = __double2float_rn(v);
    r.l = __double2float_rn(v - (double)r.h);
    return r;
}

__device__ __forceinline__ double df_to(df x) { return (double)x.h + (double)x.l; }

__device__ __forceinline__ df fast_two_sum(float a, float b)  // requires |a| >= |b| (or a == 0)
{
    df r;
    r.h = __fadd_rn(a, b);
    r.l = __fsub_rn(b, __fsub_rn(r.h, a));
    return r;
}

__device__ __forceinline__ df two_sum(float a, float b)
{
    df r;
    r.h = __fadd_rn(a, b);
    const float bb = __fsub_rn(r.h, a);
    r.l = __fadd_rn(__fsub_rn(a, __fsub_rn(r.h, bb)), __fsub_rn(b, bb));
    return r;
}

__device__ __forceinline__ df df_neg(df x) { return df_make(-x.h, -x.l); }

__device__ __forceinline__ df df_add(df x, df y)
{
    const df s = two_sum(x.h, y.h);
    return fast_two_sum(s.h, __fadd_rn(s.l, __fadd_rn(x.l, y.l)));
}

__device__ __forceinline__ df df_sub(df x, df y) { return df_add(x, df_neg(y)); }

__device__ __forceinline__ df df_mul(df x, df y)
{
    const float p = __fmul_rn(x.h, y.h);
    float e = __fmaf_rn(x.h, y.h, -p);
    e = __fmaf_rn(x.h, y.l, e);
    e = __fmaf_rn(x.l, y.h, e);
    return fast_two_sum(p, e);
}

// x times an fp32 constant c (exactly representable)
__device__ __forceinline__ df df_mulf(df x, float c)
{
    const float p = __fmul_rn(x.h, c);
    float e = __fmaf_rn(x.h, c, -p);
    e = __fmaf_rn(x.l, c, e);
    return fast_two_sum(p, e);
}

// x times a power of two (exact barring underflow)
__device__ __forceinline__ df df_scale(df x, float c) { return df_make(__fmul_rn(x.h, c), __fmul_rn(x.l, c)); }

__device__ __forceinline__ df df_sqr(df x)
{
    const float p = __fmul_rn(x.h, x.h);
    float e = __fmaf_rn(x.h, x.h, -p);
    e = __fmaf_rn(__fadd_rn(x.h, x.h), x.l, e);
    return fast_two_sum(p, e);
}

// 1 / sqrt(r) for normal r > 0 (callers keep r.h >= 2^-84): y0 from the
// special-function unit's approximate reciprocal square root, then one Newton
// step y = y0 + y0 (1 - r y0^2) / 2 with the residual formed in double-word
// precision (it is ~2^-23, so its own fp32 rounding is far below 2^-48).
__device__ __forceinline__ df df_rsqrt(df r)
{
    float y0;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(r.h));
    df y2;
    y2.h = __fmul_rn(y0, y0);
    y2.l = __fmaf_rn(y0, y0, -y2.h);
    const df ry2 = df_mul(r, y2);
    const float resid = __fsub_rn(__fsub_rn(1.0f, ry2.h), ry2.l);
    return fast_two_sum(y0, __fmul_rn(__fmul_rn(y0, 0.5f), resid));
}

// Lazily normalised accumulator of products: h collects the rounded sums and
// l the exact rounding errors of each product (two_prod) and of each addition
// (two_sum), plus the cross terms. l is only folded into h by dacc_value.
struct __align__(8) dacc {
    float h, l;
};

__device__ __forceinline__ void mac(dacc &a, const df &x, const df &y)  // a += x y
{
    const float p = __fmul_rn(x.h, y.h);
    float e = __fmaf_rn(x.h, y.h, -p);
    e = __fmaf_rn(x.h, y.l, e);
    e = __fmaf_rn(x.l, y.h, e);
    const float s = __fadd_rn(a.h, p);
    const float bb = __fsub_rn(s, a.h);
    const float err = __fadd_rn(__fsub_rn(a.h, __fsub_rn(s, bb)), __fsub_rn(p, bb));
    a.h = s;
    a.l = __fadd_rn(a.l, __fadd_rn(err, e));
}

__device__ __forceinline__ df dacc_value(const dacc &a) { return two_sum(a.h, a.l); }

// Operators, so that the generated expansion templates (P2M, L2P, ...) run in double words.
__device__ __forceinline__ df operator+(const df &x, const df &y) { return df_add(x, y); }
__device__ __forceinline__ df operator-(const df &x, const df &y) { return df_sub(x, y); }
__device__ __forceinline__ df operator-(const df &x) { return df_neg(x); }
__device__ __forceinline__ df operator*(const df &x, const df &y) { return df_mul(x, y); }
__device__ __forceinline__ df &operator+=(df &x, const df &y) { return x = df_add(x, y); }
__device__ __forceinline__ df &operator-=(df &x, const df &y) { return x = df_sub(x, y); }

using ::__shfl_xor_sync;  // keep the CUDA overloads visible next to the one below
__device__ __forceinline__ df __shfl_xor_sync(unsigned mask, df v, int o)
{
    return df_make(::__shfl_xor_sync(mask, v.h, o), ::__shfl_xor_sync(mask, v.l, o));
}

// Power-of-two units of the fp64 plans' double-word kernels: lengths in 2^ex
// with 2^(ex-1) <= the root's largest half-width < 2^ex, masses in 2^em with
// the total mass (the root's monopole) below 2^em. A node of level l then lies
// in a cell of half-size below 2^(ex - l). The scalings are exact.
__device__ __forceinline__ void df_units(const dbl4 *__restrict__ node_l, const double *__restrict__ M, int &ex,
                                         int &em)
{
    const dbl4 l = node_l[0];
    frexp(fmax(fmax(l.x, l.y), l.z), &ex);
    frexp(M[0], &em);
}

// Total degree of coefficient n in the graded coefficient order (the first
// index of degree d is d(d+1)(d+2)/6).
__host__ __device__ __forceinline__ int coef_degree(int n)
{
    return (n >= 1) + (n >= 4) + (n >= 10) + (n >= 20) + (n >= 35) + (n >= 56) + (n >= 84) + (n >= 120);
}

// x 2^e for the unit conversions: one multiplication by an exactly built power
// of two while 2^e is a normal double, the library ldexp otherwise.
__device__ __forceinline__ double scale2(double x, int e)
{
    if (e >= -1022 && e <= 1023) return x * __longlong_as_double((long long)(1023 + e) << 52);
    return ldexp(x, e);
}

// 2^k as an fp32 number, |k| <= 126
__device__ __forceinline__ float pow2f(int k) { return __int_as_float((127 + k) << 23); }

}  // namespace bfm
