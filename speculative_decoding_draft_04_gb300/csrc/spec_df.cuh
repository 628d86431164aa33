// Double-float arithmetic (a value carried as an unevaluated sum hi + lo of
// two fp32 numbers, about 48 significant bits) for the extended-precision
// re-decisions.  GB300 runs fp64 at a small fraction of its fp32 rate, so the
// re-decision path computes in pairs of fp32 instead.
//
// Every operation is written with explicitly rounded fp32 steps (no operation
// left for the compiler to contract or reorder), so this header also compiles
// as plain host C++ and gives the same results there; the CPU tests exercise
// it that way.
//
// Sources of the error-free transformations: Knuth's TwoSum, Dekker's
// FastTwoSum, TwoProduct by fused multiply-add; the exponential follows Tang's
// table-driven method (argument reduction by multiples of ln2/64, a short
// polynomial, a table of 2^(j/64)), carried out in double-float.
#pragma once

#include <string.h>

#include <math.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define SPEC_HD __host__ __device__ __forceinline__
#else
#define SPEC_HD inline
#endif

namespace spec {

struct df {
  float hi, lo;
};

SPEC_HD float rn_add(float a, float b) {
#if defined(__CUDA_ARCH__)
  return __fadd_rn(a, b);
#else
  volatile float s = a + b;
  return s;
#endif
}
SPEC_HD float rn_sub(float a, float b) {
#if defined(__CUDA_ARCH__)
  return __fsub_rn(a, b);
#else
  volatile float s = a - b;
  return s;
#endif
}
SPEC_HD float rn_mul(float a, float b) {
#if defined(__CUDA_ARCH__)
  return __fmul_rn(a, b);
#else
  volatile float s = a * b;
  return s;
#endif
}
SPEC_HD float rn_fma(float a, float b, float c) { return fmaf(a, b, c); }
SPEC_HD float rn_rcp(float a) {
#if defined(__CUDA_ARCH__)
  return __frcp_rn(a);
#else
  volatile float s = 1.0f / a;
  return s;
#endif
}

// s + e == a + b exactly (Knuth)
SPEC_HD df two_sum_df(float a, float b) {
  const float s = rn_add(a, b);
  const float bb = rn_sub(s, a);
  const float e = rn_add(rn_sub(a, rn_sub(s, bb)), rn_sub(b, bb));
  return {s, e};
}
// s + e == a + b exactly, given |a| >= |b| or a == 0 (Dekker)
SPEC_HD df fast_two_sum_df(float a, float b) {
  const float s = rn_add(a, b);
  return {s, rn_sub(b, rn_sub(s, a))};
}
// p + e == a * b exactly
SPEC_HD df two_prod_df(float a, float b) {
  const float p = rn_mul(a, b);
  return {p, rn_fma(a, b, -p)};
}

SPEC_HD df dd_add(df a, df b) {
  df s = two_sum_df(a.hi, b.hi);
  const df t = two_sum_df(a.lo, b.lo);
  s.lo = rn_add(s.lo, t.hi);
  s = fast_two_sum_df(s.hi, s.lo);
  s.lo = rn_add(s.lo, t.lo);
  return fast_two_sum_df(s.hi, s.lo);
}
SPEC_HD df dd_add_f(df a, float b) {
  df s = two_sum_df(a.hi, b);
  s.lo = rn_add(s.lo, a.lo);
  return fast_two_sum_df(s.hi, s.lo);
}
SPEC_HD df dd_neg(df a) { return {-a.hi, -a.lo}; }
SPEC_HD df dd_mul(df a, df b) {
  df p = two_prod_df(a.hi, b.hi);
  p.lo = rn_fma(a.hi, b.lo, p.lo);
  p.lo = rn_fma(a.lo, b.hi, p.lo);
  return fast_two_sum_df(p.hi, p.lo);
}
SPEC_HD df dd_mul_f(df a, float b) {
  df p = two_prod_df(a.hi, b);
  p.lo = rn_fma(a.lo, b, p.lo);
  return fast_two_sum_df(p.hi, p.lo);
}
SPEC_HD df dd_from_double(double x) {
  const float h = (float)x;
  return {h, (float)(x - (double)h)};
}
SPEC_HD double dd_to_double(df a) { return (double)a.hi + (double)a.lo; }
// a <= b, a > b (compared as exact sums)
SPEC_HD bool dd_le(df a, df b) {
  const df d = dd_add(a, dd_neg(b));
  return d.hi < 0.f || (d.hi == 0.f && d.lo <= 0.f);
}

// 1/t as a double-float: the rounded reciprocal plus one Newton correction.
SPEC_HD df dd_recip(float t) {
  const float h = rn_rcp(t);
  const float e = rn_fma(-t, h, 1.0f);         // exact residual 1 - t h
  return fast_two_sum_df(h, rn_mul(h, e));
}

// Compensated sum of fp32 terms kept as a double-float: every addition's
// rounding error is recovered exactly (TwoSum) and accumulated separately
// (the "Sum2" scheme of Ogita, Rump and Oishi, "Accurate sum and dot
// product", SIAM J. Sci. Comput. 26(6), 2005).
struct DdSum {
  float s = 0.f, c = 0.f;
  SPEC_HD void add(float x) {
    const df t = two_sum_df(s, x);
    s = t.hi;
    c = rn_add(c, t.lo);
  }
  SPEC_HD df value() const { return fast_two_sum_df(s, c); }
};

// Compensated dot product (the "Dot2" scheme of the same paper): each
// product is split exactly into p + e (TwoProd), p is added with TwoSum and
// both error terms go to the running correction, so the result is as
// accurate as a dot product evaluated in twice the working precision.
struct DdDot {
  float s = 0.f, c = 0.f;
  SPEC_HD void add(float a, float b) {
    const df p = two_prod_df(a, b);
    const df t = two_sum_df(s, p.hi);
    s = t.hi;
    c = rn_add(c, rn_add(t.lo, p.lo));
  }
  SPEC_HD df value() const { return fast_two_sum_df(s, c); }
};

// a / b in double-float: three rounded quotient digits, each from the exact
// remainder of the previous ones (long division).
SPEC_HD df dd_div(df a, df b) {
  const float rb = rn_rcp(b.hi);
  const float q1 = rn_mul(a.hi, rb);
  df rem = dd_add(a, dd_neg(dd_mul_f(b, q1)));
  const float q2 = rn_mul(rem.hi, rb);
  rem = dd_add(rem, dd_neg(dd_mul_f(b, q2)));
  const float q3 = rn_mul(rem.hi, rb);
  return dd_add_f(fast_two_sum_df(q1, q2), q3);
}

// ---------------------------------------------------------------- exponential
// Table of 2^(j/64), j = 0..63, as double-floats: entry j is the product of
// 2^(2^i/64) over the set bits i of j (binary powering from six constants,
// each the double-float nearest the exact value), so no fp64 is needed.
constexpr int DD_EXP_TAB = 64;
SPEC_HD df dd_pow2_64th(int i) {
  switch (i) {
    case 0: return {1.01088929f, -5.71160541e-09f};    // 2^(1/64)
    case 1: return {1.0218972f, -4.81155986e-08f};     // 2^(2/64)
    case 2: return {1.04427373f, 4.83347016e-08f};     // 2^(4/64)
    case 3: return {1.09050775f, -1.30775399e-08f};    // 2^(8/64)
    case 4: return {1.18920708f, 3.79763527e-08f};     // 2^(16/64)
    default: return {1.41421354f, 2.4203235e-08f};     // 2^(32/64)
  }
}
SPEC_HD void dd_exp_table_entry(df* tab, int j) {
  df v = {1.f, 0.f};
  for (int i = 0; i < 6; ++i)
    if ((j >> i) & 1) v = dd_mul(v, dd_pow2_64th(i));
  tab[j] = v;
}

// ln2 / 64 split into four parts; the first three have at most 10
// significant bits, so k * part is exact for |k| < 2^14, and the last is the
// rounded remainder (its own error times |k| stays below 1e-15).
constexpr float DD_L1 = 0.0108184814453125f;
constexpr float DD_L2 = 1.1935830116271973e-05f;
constexpr float DD_L3 = 7.414200808852911e-09f;
constexpr float DD_L4 = 6.61956471e-12f;
constexpr float DD_INV_L = 92.3324814f;                    // 64 / ln2, rounded

// e^x for a double-float x (relative error about 1e-13 for -103 < x < 88;
// returns 0 below that range: those terms are negligible next to the O(1)
// terms of every sum they enter).
SPEC_HD df dd_exp(df x, const df* tab) {
  if (!(x.hi > -103.0f)) return {0.f, 0.f};
  const float kf = rintf(rn_mul(x.hi, DD_INV_L));
  const int k = (int)kf;
  const int j = k & 63, n = (k - j) / 64;
  // r = x - k ln2/64, |r| <= ln2/128 + tiny
  const float t = rn_fma(-kf, DD_L1, x.hi);               // exact
  df r = two_sum_df(t, x.lo);
  r = dd_add_f(r, rn_mul(-kf, DD_L2));                     // products exact
  r = dd_add_f(r, rn_mul(-kf, DD_L3));
  r = dd_add_f(r, rn_mul(-kf, DD_L4));
  // e^r - 1 = r + r^2/2 + r^3 (1/6 + r/24 + r^2/120)
  const df r2 = dd_mul(r, r);
  const df h = {rn_mul(r2.hi, 0.5f), rn_mul(r2.lo, 0.5f)};
  const float tail =
      rn_mul(rn_mul(r2.hi, r.hi),
             rn_fma(r.hi, rn_fma(r.hi, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f));
  df em1 = dd_add(r, h);
  em1 = dd_add_f(em1, tail);
  const df e = dd_add_f(em1, 1.0f);
  const df v = dd_mul(e, tab[j]);
  return {ldexpf(v.hi, n), ldexpf(v.lo, n)};
}

// The logistic function 1 / (1 + e^{-z}) in double-float.  The exponential
// is always taken of -|z| (no overflow): z >= 0 gives 1/(1 + e), z < 0 gives
// e/(1 + e).  Below z = -103 the result is 0 (true value < 1.5e-45).
SPEC_HD df dd_sigmoid(df z, const df* tab) {
  const bool neg = z.hi < 0.f;
  const df e = dd_exp(neg ? z : dd_neg(z), tab);
  const df den = dd_add_f(e, 1.0f);
  return dd_div(neg ? e : df{1.0f, 0.f}, den);
}

// tanh(x) in double-float: (1 - e) / (1 + e) with e = e^{-2|x|} (no overflow),
// the sign restored.  Below |x| = 2^-5, where 1 - e would cancel, the Taylor
// series x (1 - x^2/3 + 2x^4/15 - 17x^6/315) instead (the next term is below
// 2e-14 relative; 1/3 is carried as a double-float).
SPEC_HD df dd_tanh(df x, const df* tab) {
  if (fabsf(x.hi) < 0.03125f) {
    const df t = dd_mul(x, x);
    df p = dd_add_f(dd_mul_f(t, -17.0f / 315.0f), 2.0f / 15.0f);
    p = dd_add(dd_mul(p, t), df{-0.333333343f, 9.93410776e-09f});
    return dd_add(x, dd_mul(x, dd_mul(p, t)));
  }
  const bool neg = x.hi < 0.f;
  const df ax = neg ? dd_neg(x) : x;
  const df e = dd_exp(dd_mul_f(ax, -2.0f), tab);
  const df t = dd_div(dd_add_f(dd_neg(e), 1.0f), dd_add_f(e, 1.0f));
  return neg ? dd_neg(t) : t;
}

// Bit pattern of the bfloat16 nearest (ties to even) to the finite value
// hi + lo of a normalised double-float.  hi's own rounding is right unless hi
// is exactly halfway between two bfloat16 values; then lo (|lo| < half an fp32
// ulp of hi) decides, and only lo == 0 is a true tie.
SPEC_HD uint16_t dd_to_bf16_bits(df v) {
  uint32_t u;
  memcpy(&u, &v.hi, 4);
  if ((u & 0xffffu) == 0x8000u && v.lo != 0.f) {
    const bool up = (v.lo > 0.f) == (v.hi > 0.f);          // away from zero
    return (uint16_t)((up ? u + 0x8000u : u) >> 16);
  }
  return (uint16_t)((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
}
SPEC_HD uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
}

// log(z) for a positive double-float: the fp32 logarithm plus one Newton
// step through the double-float exponential (error ~1e-14 absolute).
SPEC_HD double dd_log(df z, const df* tab) {
  const float y0 = logf(z.hi);
  const df e = dd_add_f(dd_mul(z, dd_exp(df{-y0, 0.f}, tab)), -1.0f);   // z e^{-y0} - 1
  return (double)y0 + dd_to_double(e);
}

}  // namespace spec
