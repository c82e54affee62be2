// Double-float ("fp32 pair") arithmetic for the rejection-sampling emission.
//
// A value is hi + lo with |lo| <= ulp(hi) / 2, about 48 significant bits,
// built from IEEE fp32 operations whose rounding is explicit (the __f*_rn
// intrinsics are never contracted into FMAs behind our back).  The
// error-free transformations are Knuth's TwoSum, Dekker's FastTwoSum and the
// FMA-based exact product; the exponential follows Tang's table-driven
// method ("Table-driven implementation of the exponential function in IEEE
// floating-point arithmetic", ACM TOMS 15(2), 1989), see dfx_exp2_diff.
// The fp64 value hi + lo of a pair is exact (24 + 24 bits fit in 53).
#pragma once

#include <math.h>

namespace ssv {

struct dfx {
  float hi, lo;
};

// exact a + b (Knuth's TwoSum)
__device__ __forceinline__ dfx dfx_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, err};
}

// exact a + b for |a| >= |b| or a = 0 (Dekker's FastTwoSum)
__device__ __forceinline__ dfx dfx_fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// a + b, renormalised (error <= 2^-47 |a + b| plus the inputs' own)
__device__ __forceinline__ dfx dfx_add(dfx a, dfx b) {
  const dfx s = dfx_two_sum(a.hi, b.hi);
  return dfx_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

// a * b, renormalised (the exact product of the high parts plus the cross terms)
__device__ __forceinline__ dfx dfx_mul(dfx a, dfx b) {
  const float p = __fmul_rn(a.hi, b.hi);
  const float e = __fmaf_rn(a.hi, b.hi, -p);
  const float lo = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, e));
  return dfx_fast_two_sum(p, lo);
}

__device__ __forceinline__ double dfx_to_double(dfx a) { return (double)a.hi + (double)a.lo; }

// ln 2 split into an fp32 head and tail
constexpr double kLn2d = 0.69314718055994530941723212145818;
constexpr float kLn2Hi = (float)kLn2d;
constexpr float kLn2Lo = (float)(kLn2d - (double)(float)kLn2d);

// Table of 2^(j/256), j = 0..255, in double-float, built by each CTA from
// the eight host-supplied constants pw[i] = 2^(2^i / 256): entry j is the
// product of pw[i] over the set bits i of j (at most seven double-float
// products, each within 3 * 2^-47: every entry within 1e-13).  Called by
// 256 consecutive threads (one entry each); the caller synchronises.
__device__ __forceinline__ void dfx_exp2_table(const float2* pw, float2* tab, int j) {
  dfx v{1.f, 0.f};
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if ((j >> i) & 1) v = dfx_mul(v, dfx{pw[i].x, pw[i].y});
  tab[j] = make_float2(v.hi, v.lo);
}

// 2^((l - m) * c2) for l <= m (a softmax weight relative to the row maximum
// m), c2 = log2(e) / T in double-float; tab = dfx_exp2_table.  Tang's
// table-driven reduction: x = n + j/256 + r with |r| <= 1/512, and
// 2^x = 2^n * 2^(j/256) * (1 + p), p = e^y - 1 for y = r ln 2 (|y| < 0.0014)
// formed as y + y^2 (1/2 + y/6) with y exact in double-float and the small
// quadratic part in fp32.  Relative error below 2^-46 |x| ln 2 (argument)
// + 1e-13 (table) + 2e-13 (p and the final products): 5e-13 for |x| <= 64.
// Weights below 2^-126 (and l = -inf) are returned as zero.
__device__ __forceinline__ dfx dfx_exp2_diff(float l, float m, dfx c2, const float2* tab) {
  if (!(l > -INFINITY)) return {0.f, 0.f};
  const dfx d = dfx_two_sum(l, -m);  // exact l - m <= 0
  const float xh = __fmul_rn(d.hi, c2.hi);
  const float xl = __fadd_rn(__fmaf_rn(d.hi, c2.hi, -xh), __fmaf_rn(d.hi, c2.lo, __fmul_rn(d.lo, c2.hi)));
  if (xh < -126.f) return {0.f, 0.f};
  const float k = rintf(__fmul_rn(xh, 256.f));  // xh * 256 is exact
  const int ki = (int)k;
  const int j = ki & 255;
  const int n = ki >> 8;  // floor(ki / 256)
  // xh - k/256 is exact (Sterbenz, or k = 0); r = that + xl, exactly as a pair
  const dfx r = dfx_two_sum(__fmaf_rn(k, -0.00390625f, xh), xl);
  // y = r ln 2 as yh + yl
  const float yh = __fmul_rn(r.hi, kLn2Hi);
  const float yl = __fadd_rn(__fmaf_rn(r.hi, kLn2Hi, -yh), __fmaf_rn(r.hi, kLn2Lo, __fmul_rn(r.lo, kLn2Hi)));
  // p = e^y - 1 = yh + [yh^2 (1/2 + yh/6) + yl]; |bracket| < |yh| so FastTwoSum applies
  const float q2 = __fmul_rn(__fmul_rn(yh, yh), __fmaf_rn(yh, 1.f / 6.f, 0.5f));
  const dfx pp = dfx_fast_two_sum(yh, __fadd_rn(q2, yl));
  // 2^(j/256) (1 + p) = T + T p, T >= 1 > |T p|
  const float2 t = tab[j];
  const float ph = __fmul_rn(t.x, pp.hi);
  const float lo = __fadd_rn(__fadd_rn(t.y, __fmaf_rn(t.x, pp.hi, -ph)), __fmaf_rn(t.x, pp.lo, __fmul_rn(t.y, pp.hi)));
  dfx v = dfx_fast_two_sum(t.x, ph);
  v = dfx_fast_two_sum(v.hi, __fadd_rn(v.lo, lo));
  // scale by 2^n (n >= -127 here); exact unless the low part leaves the normal range
  const float s = (n >= -126) ? __int_as_float((n + 127) << 23) : 0.f;
  return {__fmul_rn(v.hi, s), __fmul_rn(v.lo, s)};
}

}  // namespace ssv
