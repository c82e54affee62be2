// Coupled Gumbel noise generated on the device (acceptance mode
// SSV_ACCEPT_GUMBEL_GEN).
//
// SPOT review, "How it is used": drafter and target share one Gumbel noise
// value per (absolute output position, token); marginalised over the noise,
// argmax(l/T + G) is distributed as softmax(l/T) (Proposition 2).  Instead of
// reading a table, the value is generated where it is used:
//   G(seed, pos, v) = -L(-L(U)),   U = (floor(x / 2^9) + 1/2) * 2^-23,
//   x = word (v mod 4) of Philox4x32-10 at counter (floor(v / 4), pos, 0, 0)
//       under key (seed low word, seed high word),
// with L a natural logarithm evaluated by one fixed sequence of IEEE fp32
// operations (each rounded to nearest, none contracted into an FMA), so the
// value is the same bits wherever it is computed.  Philox4x32-10: Salmon,
// Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC11).
// L: argument reduction to m in [sqrt(1/2), sqrt 2] (Cody and Waite), then
// ln m = 2 atanh(s), s = (m - 1) / (m + 1), by Gregory's series to s^9.
#pragma once

#include <stdint.h>

namespace ssv {
namespace noise {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u, kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;

// fp32 constants of L, each the double value rounded once to fp32
constexpr float kSqrt2 = (float)1.41421356237309504880;
constexpr float kLn2 = (float)0.69314718055994530942;
constexpr float kC3 = (float)(2.0 / 3.0), kC5 = (float)(2.0 / 5.0), kC7 = (float)(2.0 / 7.0),
                kC9 = (float)(2.0 / 9.0);

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = kPhiloxM0 * c.x, hi0 = __umulhi(kPhiloxM0, c.x);
    const uint32_t lo1 = kPhiloxM1 * c.z, hi1 = __umulhi(kPhiloxM1, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += kPhiloxW0;
    k1 += kPhiloxW1;
  }
  return c;
}

// natural logarithm of a positive normal fp32 value (the fixed sequence)
__device__ __forceinline__ float log_f32(float x) {
  const uint32_t bits = __float_as_uint(x);
  int e = (int)((bits >> 23) & 0xFFu) - 127;
  float m = __uint_as_float((bits & 0x7FFFFFu) | 0x3F800000u);
  if (m > kSqrt2) {
    m = __fmul_rn(m, 0.5f);
    e += 1;
  }
  const float f = __fsub_rn(m, 1.f);
  const float s = __fdiv_rn(f, __fadd_rn(2.f, f));
  const float z = __fmul_rn(s, s);
  float t = __fmul_rn(kC9, z);
  t = __fmul_rn(__fadd_rn(t, kC7), z);
  t = __fmul_rn(__fadd_rn(t, kC5), z);
  t = __fmul_rn(__fadd_rn(t, kC3), z);
  const float ln1p = __fadd_rn(__fmul_rn(2.f, s), __fmul_rn(s, t));
  return __fadd_rn(__fmul_rn((float)e, kLn2), ln1p);
}

// G from the generator word x
__device__ __forceinline__ float gumbel_from_bits(uint32_t x) {
  const float u = __fmul_rn(__fadd_rn((float)(x >> 9), 0.5f), 1.1920928955078125e-07f);  // 2^-23
  return -log_f32(-log_f32(u));
}

// A cheap upper bound of gumbel_from_bits(x) (never below it): with
// U = (k + 1/2) 2^-23 and q = 2^23 - k, -ln U >= 1 - U gives
// G <= -ln(1 - U) = (23 - log2(q - 1/2)) ln 2, and log2 y >= e + (m - 1) for
// y = 2^e m, m in [1, 2).  q - 1/2 and e + (m - 1) are formed exactly from the
// bits (magic-number conversions, no int-to-float unit); 1e-3 covers the
// rounding of the fp32 evaluation of G (a few ulp of |G| <= 17) and of this
// bound's own FMA.
__device__ __forceinline__ float gumbel_upper(uint32_t x) {
  const uint32_t q1 = 0x7FFFFFu - (x >> 9);                                       // q - 1, in [0, 2^23)
  const float y = __fadd_rn(__fsub_rn(__uint_as_float(0x4B000000u | q1), 8388608.f), 0.5f);  // q - 1/2, exact
  const uint32_t yb = __float_as_uint(y);
  const float ef = __fsub_rn(__uint_as_float(0x4B000000u | (yb >> 23)), 8388735.f);   // exponent e (2^23 + 127)
  const float mf = __fsub_rn(__uint_as_float((yb & 0x7FFFFFu) | 0x3F800000u), 1.f);   // m - 1
  return __fmaf_rn(-kLn2, __fadd_rn(ef, mf), 23.f * kLn2 + 1e-3f);
}

}  // namespace noise
}  // namespace ssv
