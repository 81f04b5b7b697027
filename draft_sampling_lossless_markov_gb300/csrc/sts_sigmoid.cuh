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

#include <cuda_runtime.h>
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

// ---------------------------------------------------------------------------
// The same calibrated confidence on the fp32 pipe, in double-float arithmetic
// (pairs of fp32), for kernels that evaluate many of them on few SMs.  Relative
// error about 2^-47 |t| + 2^-46 against the exact sigmoid for |t| = |z| / tau
// <= 64; beyond, and for non-finite input, the fp64 sigmoid above.  Steps (the
// exponential by Tang's table method, "Table-driven implementation of the
// exponential function in IEEE floating-point arithmetic", ACM TOMS 1989):
//   t = z (1/tau)                 1/tau as a double-float, product exact in hi
//   |t| = n ln2/64 + r            n = rint(|t| 64/ln2), ln2/64 split in three
//                                 fp32 parts (the first with 11 bits: n times it
//                                 is exact), |r| <= ln2/128
//   e^-|t| = 2^-(n div 64) 2^-(n mod 64)/64 e^-r, the middle factor from a
//                                 64-entry double-float table, e^-r by its Taylor
//                                 series to degree 5 (the r^2 term in double-float)
//   1/(1 + w) by an approximate fp32 reciprocal y0 and the correction
//                                 y0 (1 + e + e^2), e = 1 - (1 + w) y0.
// The table T[j] = 2^(-j/64) as (hi, lo) is the caller's (sts_df_table).
// ---------------------------------------------------------------------------
namespace sts_df {
// ln2/64 = kC1 + kC2 + kC3 (kC1 has 11 significant bits: n kC1 is exact for n < 2^13)
constexpr float kC1 = 0x1.62cp-7f;
constexpr float kC2 = 0x1.217f7ep-18f;
constexpr float kC3 = -0x1.c610cap-43f;
constexpr float kInvC = 0x1.715476p+6f;  // 64/ln2, only picks n
constexpr float kDfMaxArg = 64.f;

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// |a| >= |b|
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}
__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
  p = __fmul_rn(a, b);
  e = fmaf(a, b, -p);
}

// c' = fp32(sigmoid(z / tau)); (bh, bl) = 1/tau as a double-float, rt = fp64 1/tau,
// T[j] = 2^(-j/64) as (hi, lo)
__device__ __forceinline__ float sigmoid_df(float z, float tau, float bh, float bl, double rt,
                                            const float2* __restrict__ T, float* res_hi = nullptr,
                                            float* res_lo = nullptr) {
  float th, tl;
  two_prod(z, bh, th, tl);
  tl = fmaf(z, bl, tl);
  const bool neg = th < 0.f;
  const float ah = fabsf(th), al = neg ? -tl : tl;
  if (!(ah <= kDfMaxArg)) {  // large or non-finite: the fp64 sigmoid
    if (res_hi) *res_hi = *res_lo = 0.f;
    return sts_sigmoid(z, (double)tau, rt);
  }
  const float nf = rintf(ah * kInvC);
  const int n = (int)nf;
  // r = |t| - n ln2/64 as a double-float
  const float r1 = fmaf(-nf, kC1, ah);  // exact
  float p, pe;
  two_prod(nf, kC2, p, pe);
  float rh, rl;
  two_sum(r1, -p, rh, rl);
  rl = __fadd_rn(__fsub_rn(rl, pe), __fsub_rn(al, __fmul_rn(nf, kC3)));
  fast_two_sum(rh, rl, rh, rl);
  // e^-r = 1 - r + r^2/2 + c3,  c3 = r^3 (-1/6 + r/24 - r^2/120)
  float sq, sqe;
  two_prod(rh, rh, sq, sqe);
  sqe = fmaf(2.f * rh, rl, sqe);
  const float c3 = __fmul_rn(__fmul_rn(rh, sq), fmaf(rh, fmaf(rh, -1.f / 120.f, 1.f / 24.f), -1.f / 6.f));
  float Ph, Pl, q2, q2e;
  fast_two_sum(1.f, -rh, Ph, Pl);
  fast_two_sum(Ph, 0.5f * sq, q2, q2e);
  Pl = __fadd_rn(__fadd_rn(Pl, q2e), __fadd_rn(__fsub_rn(0.5f * sqe, rl), c3));
  Ph = q2;
  // w = e^-|t| = 2^-(n>>6) T[n & 63] (Ph + Pl)
  const float2 Tj = T[n & 63];
  float wh, wl;
  two_prod(Tj.x, Ph, wh, wl);
  wl = fmaf(Tj.x, Pl, fmaf(Tj.y, Ph, wl));
  const float sc = __int_as_float((127 - (n >> 6)) << 23);  // 2^-(n>>6), n>>6 <= 92
  wh = __fmul_rn(wh, sc);
  wl = __fmul_rn(wl, sc);
  // 1 / (1 + w): y0 (1 + e + e^2) with e = 1 - (1 + w) y0
  float dh, dl;
  fast_two_sum(1.f, wh, dh, dl);
  dl = __fadd_rn(dl, wl);
  float y0;  // |1 - dh y0| <= 2^-22; the correction below absorbs it
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(dh));
  const float e = __fsub_rn(fmaf(-dh, y0, 1.f), __fmul_rn(dl, y0));
  const float ye = __fmul_rn(y0, fmaf(e, e, e));
  if (!neg) {
    if (res_hi) {
      *res_hi = y0;
      *res_lo = ye;
    }
    return __fadd_rn(y0, ye);
  }
  // w / (1 + w)
  float ph, pl;
  two_prod(wh, y0, ph, pl);
  pl = fmaf(wh, ye, fmaf(wl, y0, pl));
  if (res_hi) {
    *res_hi = ph;
    *res_lo = pl;
  }
  return __fadd_rn(ph, pl);
}


// T[j] = 2^(-j/64) as (hi, lo), j = 0..63: one entry per calling thread j
__device__ __forceinline__ float2 sts_df_table_entry(int j) {
  const double v = exp2(-(double)j / 64.0);
  const float hi = (float)v;
  return make_float2(hi, (float)(v - (double)hi));
}

// fp32(sigmoid(z / tau)) equal to the fp32 rounding of the fp64 sigmoid
// (sts_sigmoid): the double-float value is rounded unless it lies within four
// times its error bound of an fp32 rounding boundary (the midpoint between two
// neighbouring fp32 values), where the fp64 sigmoid decides instead.  Those
// cases are rare (about 1e-5 of the arguments), so the cost is the fp32
// pipe's.
__device__ __forceinline__ float sts_sigmoid_exact32(float z, float tau, float bh, float bl, double rt,
                                                     const float2* __restrict__ T) {
  float hi, lo;
  const float r = sigmoid_df(z, tau, bh, bl, rt, T, &hi, &lo);
  if (hi == 0.f && lo == 0.f) return r;  // already the fp64 sigmoid (or exactly 0)
  // residual of the rounding, (hi + lo) - r: hi - r is exact (Sterbenz)
  const float e = __fadd_rn(__fsub_rn(hi, r), lo);
  const int ex = (__float_as_int(r) >> 23) & 0xFF;
  if (ex == 0 || ex == 0xFF) return sts_sigmoid(z, (double)tau, rt);
  const float ulp = __int_as_float((ex - 23) << 23);  // ulp of r (r normal, ex >= 24 for c' > 2^-103)
  // below a power of two the gap to the next smaller fp32 value is ulp / 2
  const bool pow2 = (__float_as_int(r) & 0x7FFFFF) == 0;
  const float half = (e < 0.f && pow2) ? 0.25f * ulp : 0.5f * ulp;
  const float t = fabsf(__fmul_rn(z, bh));
  const float tol = __fmul_rn(r, fmaf(t, 0x1p-45f, 0x1p-44f));
  if (fabsf(fabsf(e) - half) <= tol) return sts_sigmoid(z, (double)tau, rt);
  return r;
}

}  // namespace sts_df

}  // namespace dspark
