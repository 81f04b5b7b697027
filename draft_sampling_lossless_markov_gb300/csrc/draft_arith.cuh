// The arithmetic of one draft probability, written once so that every kernel
// that evaluates it (logits passes, tile recompute, p_d write) rounds the same
// way.  Explicit _rn intrinsics keep the compiler from contracting a multiply
// and an add into an FMA differently in different kernels.
#pragma once

#include <cuda_runtime.h>

namespace dspark {

// 1/T for sampled rows (T > 0); greedy rows never use it
__device__ __forceinline__ float inv_temp(float T) { return T > 0.f ? __frcp_rn(T) : 1.f; }
// l = U + bias
__device__ __forceinline__ float add_base(float u, float bias) { return __fadd_rn(u, bias); }
// y = l / T
__device__ __forceinline__ float scale_logit(float l, float invT) { return __fmul_rn(l, invT); }
// exp(y - m)
__device__ __forceinline__ float exp_shifted(float y, float m) { return expf(__fsub_rn(y, m)); }
// mass of a tile with partial (m_t, s_t) relative to the row max m
__device__ __forceinline__ float tile_mass(float mt, float st, float m) { return __fmul_rn(st, expf(__fsub_rn(mt, m))); }
// p = exp(y - m) / S
__device__ __forceinline__ float prob_from(float y, float m, float S) { return __fdiv_rn(exp_shifted(y, m), S); }

}  // namespace dspark
