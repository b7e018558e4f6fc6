// hl_df.cuh -- double-float arithmetic (an unevaluated sum hi + lo of two
// fp32 values, ~48 significant bits) for the fp32-logits row kernel, and a
// 2^x built from it.
//
// GB300 runs fp64 at a small fraction of its fp32 rate, so the fp32 row
// kernel keeps its per-element arithmetic in fp32 pairs: the exponent
// argument zs - shift exactly to ~2^-44, then 2^x to ~0.3 ulp of fp32 before
// the one rounding of the gradient.  The error-free transformations are the
// classical ones (Dekker's product through an FMA, Knuth's two-sum and the
// fast two-sum when the first operand is the larger); the _rn intrinsics keep
// the compiler from contracting or reassociating them.
#pragma once
#include <stdint.h>

namespace hl {

struct DF {
    float h, l;
};

// a * b = h + l exactly
__device__ __forceinline__ DF df_two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}
// a + b = h + l exactly (any magnitudes)
__device__ __forceinline__ DF df_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}
// a + b = h + l exactly, for |a| >= |b| (or a = 0)
__device__ __forceinline__ DF df_fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// v * K - Z for an fp32 v and double-float K, Z, with an error of a few
// units of 2^-48 of the larger of |v K| and |Z|.  Not renormalised: l may
// exceed half an ulp of h (when h has cancelled), which df_exp2 absorbs.
__device__ __forceinline__ DF df_scaled_minus(float v, DF K, DF Z) {
    DF p = df_two_prod(v, K.h);
    p.l = __fmaf_rn(v, K.l, p.l);
    DF s = df_two_sum(p.h, -Z.h);
    s.l = __fadd_rn(s.l, __fsub_rn(p.l, Z.l));
    return s;
}

// Taylor coefficients of q(f) = (2^f - 1) / f = sum_{k >= 1} ln2^k f^(k-1) / k!
// (k = 2 .. 8 as fp32; ln 2 itself as a double-float), built at compile time
// from ln 2: the terms beyond k = 8 are below 2^-30 of q on |f| <= 0.52.
constexpr double DF_LN2 = 0.693147180559945309417232121458;
__host__ __device__ constexpr double df_taylor(int k) {
    double c = 1.0;
    for (int i = 1; i <= k; ++i) c = c * DF_LN2 / double(i);
    return c;
}

// 2^(a.h + a.l) = (r.h + r.l) * 2^n with r in [0.70, 1.42]: n = rint(a.h)
// (by the 1.5 * 2^23 rounding shift: |a.h| < 2^22), f = (a.h - n) + a.l,
// and 2^f = 1 + f q(f) with the polynomial's tail in fp32 and its leading
// term, the product by f and the final sum in double-float.  Relative error
// of r below 2^-25 (one rounding of f, the tail's roundings scaled by f^2).
__device__ __forceinline__ DF df_exp2(DF a, int& n) {
    constexpr float SHIFT = 12582912.f;  // 1.5 * 2^23: adding it rounds to an integer
    const float sh = __fadd_rn(a.h, SHIFT);
    const float nf = __fsub_rn(sh, SHIFT);
    n = __float_as_int(sh) - __float_as_int(SHIFT);
    const float f = __fadd_rn(__fsub_rn(a.h, nf), a.l);  // a.h - nf is exact
    constexpr float C2 = float(df_taylor(2)), C3 = float(df_taylor(3)), C4 = float(df_taylor(4)),
                    C5 = float(df_taylor(5)), C6 = float(df_taylor(6)), C7 = float(df_taylor(7)),
                    C8 = float(df_taylor(8));
    constexpr float L2H = float(DF_LN2);
    constexpr float L2L = float(DF_LN2 - double(float(DF_LN2)));
    float r = __fmaf_rn(f, C8, C7);
    r = __fmaf_rn(f, r, C6);
    r = __fmaf_rn(f, r, C5);
    r = __fmaf_rn(f, r, C4);
    r = __fmaf_rn(f, r, C3);
    r = __fmaf_rn(f, r, C2);
    const float u = __fmul_rn(f, r);                  // |u| <= 0.13
    DF q = df_fast_two_sum(L2H, u);                   // q = ln2 + u
    q.l = __fadd_rn(q.l, L2L);
    DF t = df_two_prod(f, q.h);                       // t = f q
    t.l = __fmaf_rn(f, q.l, t.l);
    DF e = df_fast_two_sum(1.f, t.h);                 // 1 + t, |t| <= 0.42
    e.l = __fadd_rn(e.l, t.l);
    return e;
}

// 2^n as an fp32 for -126 <= n <= 127 (exact)
__device__ __forceinline__ float df_pow2i(int n) { return __int_as_float((n + 127) << 23); }

}  // namespace hl

namespace hl {

// 2^n as an fp64 for -1022 <= n <= 1023 (exact)
__device__ __forceinline__ double df_pow2d(int n) {
    return __longlong_as_double((long long)(n + 1023) << 52);
}

// 2^x for an fp64 x (|x| < 2^22) through df_exp2: relative error below 2^-25
// and below |x| 2^-25 for small |x| (2^0 is exactly 1); 0 below 2^-1022.
__device__ __forceinline__ double df_exp2d(double x) {
    const float h = float(x);
    int n;
    const DF e = df_exp2({h, float(x - double(h))}, n);
    if (n < -1000) return 0.0;
    return (double(e.h) + double(e.l)) * df_pow2d(n);
}

// log2(x) for an fp64 x > 0 (normal): y0 = log2f(x) in fp32, then one
// correction y = y0 + log2(1 + m) with 1 + m = x 2^-y0 formed in fp64 and
// log2(1 + m) = (m - m^2 / 2) log2(e) (|m| ~ 2^-20: the cubic term is below
// 2^-60).  The error is that of 2^-y0: below 2^-25 / ln2 absolute, and below
// |y0| 2^-25 / ln2 near x = 1 (where the result itself is small).
__device__ __forceinline__ double df_log2d(double x) {
    const float y0 = log2f(float(x));
    int n;
    const DF e = df_exp2({-y0, 0.f}, n);
    const double m = x * ((double(e.h) + double(e.l)) * df_pow2d(n)) - 1.0;
    constexpr double LOG2E = 1.0 / DF_LN2;
    return double(y0) + (m - 0.5 * m * m) * LOG2E;
}

// 1 / v for an fp64 v > 0 (normal, within fp32's range): fp32 reciprocal,
// then two Newton steps in fp64 (2^-23 -> 2^-46 -> below fp64 rounding).
__device__ __forceinline__ double df_recipd(double v) {
    double r = double(__frcp_rn(float(v)));
    r = r * (2.0 - v * r);
    r = r * (2.0 - v * r);
    return r;
}

}  // namespace hl
