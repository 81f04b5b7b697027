// Calibrated confidence c' = fp32(sigmoid(z / tau)) with the sigmoid in fp64.
//
// [DSpark] 方法细节, "事后校准（Post-hoc Calibration）": Sequential Temperature
// Scaling divides each position's confidence logit by a per-position
// temperature.  c' feeds sort keys and calibration bins, so it is the fp32
// rounding of an fp64 evaluation; the fp64 sigmoid here is written out (no
// library exp) so that its cost is a known count of fp64 operations:
//
//   t = z / tau            z * (1/tau), then one exact-residual correction (3 ops)
//   w = e^-|t|             Cody-Waite reduction |t| = n ln2 - r with a split ln2
//                          (Cody & Waite, "Software Manual for the Elementary
//                          Functions", 1980), e^r by its Taylor series to degree
//                          13 in Horner form (|r| <= 0.35: truncation < 2^-56),
//                          times 2^-n built from exponent bits  (19 ops)
//   q = 1 / (1 + w)        fp32 reciprocal seed, two Newton steps  (5 ops)
//   sigmoid(t) = q (t >= 0) or w q (t < 0)                          (1 op)
//
// 28 fp64 arithmetic operations in all, plus four fp64 <-> fp32 / int
// conversions.
//
// The result is within a few fp64 ulps of the exact sigmoid, so its fp32
// rounding is the correctly rounded value except when the exact sigmoid lies
// within ~1e-15 (relative) of an fp32 rounding midpoint.  |t| is capped at 110:
// beyond it the fp32 result is already 1 (t > 0) or 0 (t < 0).
#pragma once

#include <stdint.h>

namespace dspark {

namespace sts_detail {
// ln 2 = kLn2Hi + kLn2Lo; kLn2Hi holds 42 significant bits, so n * kLn2Hi is
// exact for |n| < 2^11
constexpr double kLn2Hi = 0x1.62e42fefa38p-1;
constexpr double kLn2Lo = 0x1.ef35793c7673p-45;
constexpr double kLog2e = 0x1.71547652b82fep+0;
constexpr double kMaxArg = 110.0;
}  // namespace sts_detail

// 1/k! for k = 0..13, correctly rounded
__device__ __forceinline__ double sts_inv_fact(int k) {
  constexpr double f[14] = {1.0,
                            1.0,
                            1.0 / 2.0,
                            1.0 / 6.0,
                            1.0 / 24.0,
                            1.0 / 120.0,
                            1.0 / 720.0,
                            1.0 / 5040.0,
                            1.0 / 40320.0,
                            1.0 / 362880.0,
                            1.0 / 3628800.0,
                            1.0 / 39916800.0,
                            1.0 / 479001600.0,
                            1.0 / 6227020800.0};
  return f[k];
}

// c' for logit z, temperature tau (> 0) and rtau = fp64(1 / tau)
__device__ __forceinline__ float sts_sigmoid(float z, double tau, double rtau) {
  using namespace sts_detail;
  const double zd = (double)z;
  double t = zd * rtau;
  const double res = fma(-t, tau, zd);  // z - t tau, exact
  t = fma(res, rtau, t);
  const double a = fmin(fabs(t), kMaxArg);
  const double kd = rint(a * kLog2e);
  double r = fma(kd, kLn2Hi, -a);  // exact (Sterbenz)
  r = fma(kd, kLn2Lo, r);          // r = n ln2 - a, |r| <= 0.35
  double p = sts_inv_fact(13);
#pragma unroll
  for (int k = 12; k >= 0; --k) p = fma(p, r, sts_inv_fact(k));
  const int n = (int)kd;  // 0..159
  const double w = p * __longlong_as_double((long long)(1023 - n) << 52);  // e^-a
  const double d = 1.0 + w;                                                  // (1, 2]
  float seed;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(seed) : "f"((float)d));
  double q = (double)seed;
  double e = fma(-d, q, 1.0);
  q = fma(q, e, q);
  e = fma(-d, q, 1.0);
  q = fma(q, e, q);
  return (float)(t >= 0.0 ? q : w * q);
}

}  // namespace dspark
