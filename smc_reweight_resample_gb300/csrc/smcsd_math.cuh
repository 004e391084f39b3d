// smcsd_math.cuh -- double-float ("dd": an unevaluated sum hi + lo of two float32) arithmetic
// and a double-float exponential, for the rows that are sampled by inverse CDF.
//
// Why: an inverse-CDF draw over a 128K-token vocabulary compares u*R with prefix sums whose
// steps are ~1e-7 of the total. Float32 exp (a relative error of ~1e-7 per term) moves those
// prefix sums by about one step and changes ~1e-4 of all draws; a per-term relative error near
// 1e-12 makes such changes vanishingly rare. The streaming normalisers (logsumexp) do not need
// this and use the hardware exp2.
//
// Error-free transformations: Knuth's two-sum, Dekker's fast-two-sum, and the FMA-based exact
// product. The exponential follows Tang's table-driven method (P. T. P. Tang, "Table-driven
// implementation of the exponential function in IEEE floating-point arithmetic", ACM TOMS 15(2),
// 1989): x*log2(e) = n + j/32 + g with an integer n, j in [0,32) and |g| <= 1/64; then
// exp(x) = 2^n * 2^(j/32) * exp(g*ln 2), the middle factor from a 32-entry double-float table and
// the last from a short Taylor series. The table is filled on the host from the C library's
// double exp2 (see make_exp2_table()).
//
// Every function is host+device so the same code can be checked on the CPU. On the device the
// float operations go through the IEEE round-to-nearest intrinsics (__fadd_rn and friends), which
// the compiler never contracts into FMAs; host builds must use -ffp-contract=off.
#pragma once

#include <math.h>
#include <stdint.h>

#ifdef __CUDACC__
#define SMCSD_HD __host__ __device__ __forceinline__
#else
#define SMCSD_HD static inline
#endif

namespace smcsd {

SMCSD_HD float f_add(float a, float b) {
#ifdef __CUDA_ARCH__
    return __fadd_rn(a, b);
#else
    return a + b;
#endif
}
SMCSD_HD float f_sub(float a, float b) {
#ifdef __CUDA_ARCH__
    return __fsub_rn(a, b);
#else
    return a - b;
#endif
}
SMCSD_HD float f_mul(float a, float b) {
#ifdef __CUDA_ARCH__
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}
SMCSD_HD float f_fma(float a, float b, float c) {
#ifdef __CUDA_ARCH__
    return __fmaf_rn(a, b, c);
#else
    return fmaf(a, b, c);
#endif
}
SMCSD_HD float f_div(float a, float b) {
#ifdef __CUDA_ARCH__
    return __fdiv_rn(a, b);
#else
    return a / b;
#endif
}

struct dd {
    float hi, lo;
};

// Knuth two-sum: s + e == a + b exactly.
SMCSD_HD dd two_sum(float a, float b) {
    float s = f_add(a, b);
    float bb = f_sub(s, a);
    float e = f_add(f_sub(a, f_sub(s, bb)), f_sub(b, bb));
    return {s, e};
}
// Dekker fast-two-sum: exact when |a| >= |b| (or a == 0).
SMCSD_HD dd fast_two_sum(float a, float b) {
    float s = f_add(a, b);
    float e = f_sub(b, f_sub(s, a));
    return {s, e};
}
// p + e == a * b exactly (barring underflow).
SMCSD_HD dd two_prod(float a, float b) {
    float p = f_mul(a, b);
    float e = f_fma(a, b, -p);
    return {p, e};
}
// Accurate double-float sum (both parts through two-sum), normalised.
SMCSD_HD dd dd_add(dd a, dd b) {
    dd s = two_sum(a.hi, b.hi);
    dd t = two_sum(a.lo, b.lo);
    s.lo = f_add(s.lo, t.hi);
    s = fast_two_sum(s.hi, s.lo);
    s.lo = f_add(s.lo, t.lo);
    return fast_two_sum(s.hi, s.lo);
}
SMCSD_HD dd dd_neg(dd a) { return {-a.hi, -a.lo}; }
SMCSD_HD dd dd_sub(dd a, dd b) { return dd_add(a, dd_neg(b)); }
SMCSD_HD dd dd_mul(dd a, dd b) {
    dd p = two_prod(a.hi, b.hi);
    p.lo = f_fma(a.hi, b.lo, p.lo);
    p.lo = f_fma(a.lo, b.hi, p.lo);
    return fast_two_sum(p.hi, p.lo);
}
SMCSD_HD dd dd_mul_f(dd a, float b) {
    dd p = two_prod(a.hi, b);
    p.lo = f_fma(a.lo, b, p.lo);
    return fast_two_sum(p.hi, p.lo);
}
// 1/a by one Newton step from the float reciprocal.
SMCSD_HD dd dd_recip(dd a) {
    float r0 = f_div(1.0f, a.hi);
    dd ar = dd_mul_f(a, r0);
    dd e = dd_sub(dd{1.0f, 0.0f}, ar);
    dd c = dd_mul_f(e, r0);
    return dd_add(dd{r0, 0.0f}, c);
}
// a / b by long division on the float quotient: q1 = a.hi / b.hi, then two correction digits
// from the exact remainders a - q1 b and a - (q1 + q2) b. A quotient that is a float (25 / 5) comes
// out exact, so that a ratio compared with a threshold it equals is not off by the last digit.
SMCSD_HD dd dd_div(dd a, dd b) {
    const float q1 = f_div(a.hi, b.hi);
    dd r = dd_sub(a, dd_mul_f(b, q1));
    const float q2 = f_div(r.hi, b.hi);
    r = dd_sub(r, dd_mul_f(b, q2));
    const float q3 = f_div(r.hi, b.hi);
    const dd q = fast_two_sum(q1, q2);
    return dd_add(q, dd{q3, 0.0f});
}
// a > b for normalised double-floats.
SMCSD_HD bool dd_gt(dd a, dd b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
SMCSD_HD double dd_to_double(dd a) { return (double)a.hi + (double)a.lo; }

// 2^k for an integer k in [-126, 127] as a float, built from its exponent field; 0 below -126.
SMCSD_HD float pow2i(int k) {
    int e = k + 127;
    e = e < 0 ? 0 : (e > 254 ? 254 : e);
    union {
        uint32_t u;
        float f;
    } v;
    v.u = ((uint32_t)e) << 23;
    return v.f;
}

// 2^(j/32), j = 0..31, as double-floats.
struct Exp2Table {
    float hi[32];
    float lo[32];
};

// Host: fill the 2^(j/32) table from the C library's double exp2 (error below 1e-16).
static inline Exp2Table make_exp2_table() {
    Exp2Table T;
    for (int j = 0; j < 32; ++j) {
        double v = exp2((double)j / 32.0);
        float h = (float)v;
        T.hi[j] = h;
        T.lo[j] = (float)(v - (double)h);
    }
    return T;
}

// A value (hi + lo) * 2^n with hi in [1, 2): the result of exp_split.
struct ddx {
    float hi, lo;
    int n;
};

// log2(e) and ln(2) as double-floats (high parts exact in float, low parts the float rounding
// of the remainder).
#define SMCSD_LOG2E_HI 1.44269502162933349609375f
#define SMCSD_LOG2E_LO 1.925963033500011079e-08f
#define SMCSD_LN2_HI 0.693147182464599609375f
#define SMCSD_LN2_LO (-1.9046542121259336e-09f)

// exp(x) for a double-float x with |x| <= 65536, as (hi + lo) * 2^n with hi in [1,2).
// Relative error ~1e-13 for |x| <= 100, growing like |x| * 2^-48 beyond.
SMCSD_HD ddx exp_split(dd x, const Exp2Table& T) {
    // t = x * log2(e) in double-float
    dd t = dd_mul(x, dd{SMCSD_LOG2E_HI, SMCSD_LOG2E_LO});
    // t = n0 + f with n0 = rint(t.hi): t.hi - n0 is exact (Sterbenz), |f| <= 1/2 + tiny
    float n0 = rintf(t.hi);
    dd f = two_sum(f_sub(t.hi, n0), t.lo);
    // f = j/32 + g, j = rint(32 f) in [-16, 16], |g| <= 1/64 + tiny (the subtraction is exact)
    float jf = rintf(f_mul(f.hi, 32.0f));
    dd g = two_sum(f_sub(f.hi, f_mul(jf, 0.03125f)), f.lo);
    int j = (int)jf;
    int n = (int)n0 + (j >> 5);  // arithmetic shift: -1 for j < 0
    j &= 31;
    dd y = dd_mul(g, dd{SMCSD_LN2_HI, SMCSD_LN2_LO});  // |y| < 0.011
    // exp(y) - 1 = y + y^2/2 + y^3/6 + ... ; y^2 carried exactly in its high part
    dd sq = two_prod(y.hi, y.hi);
    float yh = y.hi;
    float tail = f_mul(f_mul(sq.hi, yh),
                       f_fma(yh, f_fma(yh, f_fma(yh, f_fma(yh, 1.9841269841e-4f, 1.3888888889e-3f),
                                                 8.3333333333e-3f),
                                       4.1666666667e-2f),
                             1.6666666667e-1f));
    dd s = two_sum(yh, f_mul(sq.hi, 0.5f));
    float small = f_add(f_add(y.lo, f_mul(f_fma(f_mul(2.0f, yh), y.lo, sq.lo), 0.5f)), tail);
    s.lo = f_add(s.lo, small);
    dd e = two_sum(1.0f, s.hi);
    e.lo = f_add(e.lo, s.lo);
    dd r = dd_mul(dd{T.hi[j], T.lo[j]}, e);  // in (0.98, 1.98)
    if (r.hi >= 2.0f) {
        r.hi = f_mul(r.hi, 0.5f);
        r.lo = f_mul(r.lo, 0.5f);
        n += 1;
    } else if (r.hi < 1.0f) {
        r.hi = f_mul(r.hi, 2.0f);
        r.lo = f_mul(r.lo, 2.0f);
        n -= 1;
    }
    return {r.hi, r.lo, n};
}

}  // namespace smcsd
