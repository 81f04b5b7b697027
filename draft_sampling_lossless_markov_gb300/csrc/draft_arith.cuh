// The arithmetic of one probability, written once so that every kernel that
// evaluates it (draft logits passes, tile recompute, p_d write, verify row
// statistics, residual) rounds the same way.  Explicit _rn intrinsics keep the
// compiler from contracting a multiply and an add into an FMA differently in
// different kernels.
//
// softmax(l / T) is evaluated in base 2: with c = log2(e) / T,
//     y = l * c,   m = max y,   w = 2^(y - m),   S = sum w,   p = w * (1 / S)
// which equals exp(l/T - max l/T) / sum exp(...) up to fp32 rounding.
#pragma once

#include <cuda_runtime.h>

namespace dspark {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)

// c = log2(e) / T for sampled rows (T > 0); 1 for greedy rows, whose argmax is
// then taken on the logits themselves (a scale could merge two distinct logits)
__device__ __forceinline__ float row_scale(float T) { return T > 0.f ? __fmul_rn(__frcp_rn(T), kLog2e) : 1.f; }
// l = U + bias
__device__ __forceinline__ float add_base(float u, float bias) { return __fadd_rn(u, bias); }
// y = l * c
__device__ __forceinline__ float scale_logit(float l, float c) { return __fmul_rn(l, c); }
// 2^x by the hardware's approximate base-2 exponential (relative error about
// 2^-22; results below 2^-126 flush to zero, far under every probability
// tolerance of the library)
__device__ __forceinline__ float ex2_ftz(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// 2^(y - m)
__device__ __forceinline__ float exp_shifted(float y, float m) { return ex2_ftz(__fsub_rn(y, m)); }
// mass of a tile with partial (m_t, s_t) relative to the row max m
__device__ __forceinline__ float tile_mass(float mt, float st, float m) { return __fmul_rn(st, ex2_ftz(__fsub_rn(mt, m))); }
// 2^(l c - m) with l c - m formed by one fma (one rounding instead of two): the
// fused-sweep kernel's form, used by every step of that kernel that weighs a
// logit (chunk sums, the crossing chunk's walk, the p_d rows), so that they
// agree with each other
__device__ __forceinline__ float exp_scaled(float l, float c, float m) { return ex2_ftz(__fmaf_rn(l, c, -m)); }
// 1 / S
__device__ __forceinline__ float inv_sum(float S) { return __frcp_rn(S); }
// p = 2^(y - m) / S, as 2^(y - m) * (1 / S)
__device__ __forceinline__ float prob_from(float y, float m, float invS) { return __fmul_rn(exp_shifted(y, m), invS); }

}  // namespace dspark
