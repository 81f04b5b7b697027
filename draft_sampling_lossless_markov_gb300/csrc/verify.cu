// Lossless rejection-sampling verification.
//
// [DSpark] 背景知识与设计原则, "投机解码的延迟建模": accept x_k with probability
// min(1, p_t^k(x_k) / p_d^k(x_k)), left to right, the first rejection discards
// the rest.  [MTP Survey] §2.2 "拒绝采样": resample the rejecting position from
// norm(max(0, p_t - p_d)); bonus token when everything is accepted; argmax
// compare at temperature 0.
//
// k_verify_rowstats  one CTA per slice of a kept row (request r, row j <= l_r):
//                    max and sum of 2^(z c) (sampled) or argmax of z (greedy)
// k_verify_finish    one CTA per request: the accept tests of all positions in
//                    one warp (p_t at each draft token from the combined row
//                    statistics), the first rejection, then one inverse-CDF draw
//                    over the final row (residual or bonus): per-chunk sums in
//                    shared memory, then a re-read of the one chunk that holds
//                    the draw.
#include "common.cuh"
#include "draft_arith.cuh"
#include "internal.h"

namespace dspark {

constexpr int RS_THREADS = 256;
constexpr int FIN_THREADS = 1024;

// Each kept row is split into RS_PARTS contiguous slices, one CTA per slice, so
// that the grid is many small CTAs instead of one wave of big ones plus a
// nearly empty second wave.  Partial per (row, slice): sampled rows store
// (max y, sum 2^(y - max)); greedy rows store (argmax value, argmax index).
template <typename T>
__global__ void __launch_bounds__(RS_THREADS) k_verify_rowstats(const T* __restrict__ target,
                                                                const int32_t* __restrict__ offsets,
                                                                const int32_t* __restrict__ ell,
                                                                const float* __restrict__ temp, int V,
                                                                float4* __restrict__ rsp) {
  __shared__ float sm_a[RS_THREADS / 32], sm_b[RS_THREADS / 32];
  __shared__ int sm_i[RS_THREADS / 32];
  const int r = blockIdx.x, j = blockIdx.y, part = blockIdx.z;
  const int L = ell[r];
  if (j > L) return;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const size_t row = (size_t)offsets[r] + j;
  const T* z = target + row * V;
  const float T_ = temp[r];
  const bool sampled = T_ > 0.f;
  const float c = row_scale(T_);
  const bool vec = (V & 7) == 0;
  const int span = ((V + RS_PARTS - 1) / RS_PARTS + 7) & ~7;  // multiple of 8: vector loads stay aligned
  const int lo = min(part * span, V), hi = min(lo + span, V);

  if (sampled) {
    float m = -INFINITY, s = 0.f;
    if (vec) {
      for (int i = lo + tid * 8; i < hi; i += RS_THREADS * 8) {
        float v[8];
        load8_stream(z + i, v);
        float lm = -INFINITY;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          v[e] = scale_logit(v[e], c);
          lm = fmaxf(lm, v[e]);
        }
        if (lm > m) {
          s = s * exp2f(m - lm);
          m = lm;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) s += exp_shifted(v[e], m);
      }
    } else {
      for (int i = lo + tid; i < hi; i += RS_THREADS) {
        const float y = scale_logit(to_f32(z[i]), c);
        if (y > m) {
          s = s * exp2f(m - y);
          m = y;
        }
        s += exp_shifted(y, m);
      }
    }
    warp_lse(m, s);
    if (lane == 0) {
      sm_a[wid] = m;
      sm_b[wid] = s;
    }
    __syncthreads();
    if (tid == 0) {
      float M = sm_a[0], S = sm_b[0];
      for (int w_ = 1; w_ < RS_THREADS / 32; ++w_) lse_merge(M, S, sm_a[w_], sm_b[w_]);
      rsp[row * RS_PARTS + part] = make_float4(M, S, 0.f, 0.f);
    }
  } else {
    float av = -INFINITY;
    int ai = INT_MAX;
    if (vec) {
      for (int i = lo + tid * 8; i < hi; i += RS_THREADS * 8) {
        float v[8];
        load8_stream(z + i, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) argmax_merge(av, ai, v[e], i + e);
      }
    } else {
      for (int i = lo + tid; i < hi; i += RS_THREADS) argmax_merge(av, ai, to_f32(z[i]), i);
    }
    warp_argmax(av, ai);
    if (lane == 0) {
      sm_a[wid] = av;
      sm_i[wid] = ai;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w_ = 1; w_ < RS_THREADS / 32; ++w_) argmax_merge(av, ai, sm_a[w_], sm_i[w_]);
      rsp[row * RS_PARTS + part] = make_float4(av, __int_as_float(ai), 0.f, 0.f);
    }
  }
}

// Row statistics from the slice partials, combined in slice order:
// sampled rows -> (M, S) of the whole row; greedy rows -> argmax (in .z).
__device__ __forceinline__ float4 row_stats(const float4* __restrict__ rsp, size_t row, bool sampled) {
  const float4 p0 = rsp[row * RS_PARTS];
  if (sampled) {
    float M = p0.x, S = p0.y;
    for (int q = 1; q < RS_PARTS; ++q) {
      const float4 pq = rsp[row * RS_PARTS + q];
      lse_merge(M, S, pq.x, pq.y);
    }
    return make_float4(M, S, __int_as_float(-1), 0.f);
  }
  float av = p0.x;
  int ai = __float_as_int(p0.y);
  for (int q = 1; q < RS_PARTS; ++q) {
    const float4 pq = rsp[row * RS_PARTS + q];
    argmax_merge(av, ai, pq.x, __float_as_int(pq.y));
  }
  return make_float4(0.f, 1.f, __int_as_float(ai), 0.f);
}

// q(v) of the final draw: residual max(0, p_t - p_d) or the bonus weight 2^(y - m)
template <typename T, int MODE>  // MODE 0: residual, 1: target weights
__device__ __forceinline__ float final_weight(const T* z, const float* pd, int v, float c, float m, float invS) {
  const float y = scale_logit(to_f32(z[v]), c);
  if (MODE == 1) return exp_shifted(y, m);
  return fmaxf(0.f, __fsub_rn(prob_from(y, m, invS), pd[v]));
}

// Chunks of 256 tokens (8 per lane) per warp segment; a segment holds at most
// FIN_MAXCH of them, so V <= 32 * 256 * FIN_MAXCH = DSPARK_MAX_VOCAB.
constexpr int FIN_MAXCH = 256;

// q of the 8 tokens v0..v0+7 (masked past hi), with vector loads when the row
// allows them; both branches evaluate final_weight's formula
template <typename T, int MODE>
__device__ __forceinline__ void chunk_weights(const T* z, const float* pd, int v0, int hi, bool vec, float c, float m,
                                              float invS, float (&q)[8]) {
  if (vec && v0 + 8 <= hi) {
    float zv[8], pv[8];
    load8(z + v0, zv);
    if (MODE == 0) load8(pd + v0, pv);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float y = scale_logit(zv[e], c);
      q[e] = (MODE == 1) ? exp_shifted(y, m) : fmaxf(0.f, __fsub_rn(prob_from(y, m, invS), pv[e]));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) q[e] = (v0 + e < hi) ? final_weight<T, MODE>(z, pd, v0 + e, c, m, invS) : 0.f;
  }
}

__device__ __forceinline__ float lane_sum8(const float (&q)[8]) {
  return ((q[0] + q[1]) + (q[2] + q[3])) + ((q[4] + q[5]) + (q[6] + q[7]));
}

// One CTA draws a token from the unnormalised weights q over the row by
// inverse CDF in token order: the sum runs over 32 warp segments, each a
// sequence of 256-token chunks.  Pass 1 records every chunk's total in shared
// memory (loads of consecutive chunks overlap); the warp whose segment holds
// u * sum then finds the chunk from those totals and re-reads only that chunk
// to find the token.  Rounding that leaves no crossing falls back to the last
// token with positive weight of the chosen segment or chunk.
template <typename T, int MODE>
__device__ int final_draw(const T* z, const float* pd, int V, float c, float m, float invS, float u, float* tot,
                          float* sm_seg, int* sm_int, float* sm_flt, bool& zero_mass) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int NW = FIN_THREADS / 32;
  const int seg = (((V + NW - 1) / NW) + 255) & ~255;
  const int s_lo = min(wid * seg, V), s_hi = min(s_lo + seg, V);
  const int nch = (s_hi - s_lo + 255) >> 8;
  const bool vec = (V & 7) == 0;
  float acc = 0.f;
#pragma unroll 4
  for (int ci = 0; ci < nch; ++ci) {
    float q[8];
    chunk_weights<T, MODE>(z, pd, s_lo + ci * 256 + lane * 8, s_hi, vec, c, m, invS, q);
    const float ct = warp_sum(lane_sum8(q));
    if (lane == 0) tot[wid * FIN_MAXCH + ci] = ct;
    acc += ct;
  }
  if (lane == 0) sm_seg[wid] = acc;
  __syncthreads();
  if (wid == 0) {
    const float sv = sm_seg[lane];
    const float incl = warp_inclusive_scan(sv);
    const float total = __shfl_sync(0xffffffffu, incl, 31);
    const float target = u * total;
    const unsigned over = __ballot_sync(0xffffffffu, incl > target);
    const unsigned pos = __ballot_sync(0xffffffffu, sv > 0.f);
    const bool hit = over != 0u && total > 0.f;
    const int w_star = hit ? __ffs(over) - 1 : (pos ? 31 - __clz(pos) : 0);
    float pre = __shfl_up_sync(0xffffffffu, incl, 1);
    pre = __shfl_sync(0xffffffffu, (lane == 0) ? 0.f : pre, w_star);
    if (lane == 0) {
      sm_int[0] = w_star;
      sm_int[1] = hit;
      sm_flt[0] = pre;
      sm_flt[1] = target;
      sm_flt[2] = total;
    }
  }
  __syncthreads();
  zero_mass = !(sm_flt[2] > 0.f);
  const int w_star = sm_int[0];
  const bool hit = sm_int[1] != 0;
  if (wid == w_star) {
    const int g_lo = min(w_star * seg, V), g_hi = min(g_lo + seg, V);
    const int gch = (g_hi - g_lo + 255) >> 8;
    const float target = sm_flt[1];
    float run = sm_flt[0];
    int cstar = -1, lastc = -1;
    float cpre = 0.f;
    for (int c0 = 0; c0 < gch; c0 += 32) {
      const int ci = c0 + lane;
      const float tv = ci < gch ? tot[w_star * FIN_MAXCH + ci] : 0.f;
      const float incl = warp_inclusive_scan(tv);
      const unsigned over = __ballot_sync(0xffffffffu, hit && run + incl > target);
      const unsigned pos = __ballot_sync(0xffffffffu, tv > 0.f);
      if (pos) lastc = c0 + 31 - __clz(pos);
      float excl = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) excl = 0.f;
      if (over) {
        const int Lc = __ffs(over) - 1;
        cstar = c0 + Lc;
        cpre = run + __shfl_sync(0xffffffffu, excl, Lc);
        break;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    const bool in_chunk = cstar >= 0;
    if (!in_chunk) cstar = lastc;
    int x = -1;
    if (cstar >= 0) {
      float q[8];
      const int v0 = g_lo + cstar * 256 + lane * 8;
      chunk_weights<T, MODE>(z, pd, v0, g_hi, vec, c, m, invS, q);
      const float ls = lane_sum8(q);
      const float incl = warp_inclusive_scan(ls);
      int lastp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (q[e] > 0.f) lastp = v0 + e;
      if (in_chunk) {
        const unsigned over = __ballot_sync(0xffffffffu, cpre + incl > target);
        if (over) {
          const int Ll = __ffs(over) - 1;
          float pre = __shfl_up_sync(0xffffffffu, incl, 1);
          pre = __shfl_sync(0xffffffffu, (lane == 0) ? 0.f : pre, Ll);
          int xl = -1;
          if (lane == Ll) {
            float a = cpre + pre;
            for (int e = 0; e < 8; ++e) {
              a += q[e];
              if (a > target) {
                xl = v0 + e;
                break;
              }
            }
            if (xl < 0) xl = lastp;
          }
          x = __shfl_sync(0xffffffffu, xl, Ll);
        }
      }
      if (x < 0) {  // rounding left no crossing: last positive weight of the chunk
        int lp = lastp;
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
        x = lp;
      }
    }
    if (lane == 0) sm_int[2] = x;
  }
  __syncthreads();
  const int x = sm_int[2];
  __syncthreads();
  return x;
}

template <typename T>
__global__ void __launch_bounds__(FIN_THREADS) k_verify_finish(const T* __restrict__ target,
                                                               const int32_t* __restrict__ offsets,
                                                               const int32_t* __restrict__ ell,
                                                               const int32_t* __restrict__ tokens,
                                                               const float* __restrict__ pd_rows,
                                                               const float* __restrict__ pd_tok,
                                                               const float* __restrict__ temp,
                                                               const uint32_t* __restrict__ req_id, uint64_t seed,
                                                               int G, int V, const float4* __restrict__ rs,
                                                               int32_t* __restrict__ n_accept,
                                                               int32_t* __restrict__ out_tok,
                                                               int32_t* __restrict__ n_out, WsHeader* hdr) {
  __shared__ float tot[32 * FIN_MAXCH];
  __shared__ float sm_seg[32];
  __shared__ int sm_int[4];
  __shared__ float sm_flt[4];
  __shared__ int s_m;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  const int L = ell[r];
  const float T_ = temp[r];
  const bool sampled = T_ > 0.f;
  const uint32_t req = req_id[r];
  const int base = offsets[r];
  if (tid < 32) {
    // the accept tests of positions 1..L in parallel (gamma <= 32); the first
    // rejection ends the accepted prefix
    const int j = tid;
    bool acc = true;
    if (j < L) {
      const size_t row = (size_t)base + j;
      const float4 st = row_stats(rs, row, sampled);
      int x = tokens[(size_t)r * G + j];
      if (x < 0 || x >= V) {
        report_error(hdr, DSPARK_BAD_INPUT, x);
        x = 0;
      }
      if (sampled) {
        const float c = row_scale(T_);
        const float ptok = prob_from(scale_logit(to_f32(target[row * V + x]), c), st.x, inv_sum(st.y));
        const float u = philox_uniform(seed, req, (uint32_t)(j + 1), 1u);
        acc = __fmul_rn(u, pd_tok[(size_t)r * G + j]) < ptok;
      } else {
        acc = x == __float_as_int(st.z);
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, !acc);
    if (tid == 0) s_m = rej ? __ffs(rej) - 1 : L;
  }
  __syncthreads();
  const int m = s_m;
  for (int i = tid; i <= G; i += FIN_THREADS) out_tok[(size_t)r * (G + 1) + i] = (i < m) ? tokens[(size_t)r * G + i] : -1;
  const float4 st = row_stats(rs, (size_t)base + m, sampled);
  int x;
  if (!sampled) {
    x = __float_as_int(st.z);
  } else {
    const T* z = target + ((size_t)base + m) * V;
    const float c = row_scale(T_);
    bool zero_mass = false;
    if (m < L) {
      const float u = philox_uniform(seed, req, (uint32_t)(m + 1), 2u);
      const float* pd = pd_rows + ((size_t)r * G + m) * V;
      x = final_draw<T, 0>(z, pd, V, c, st.x, inv_sum(st.y), u, tot, sm_seg, sm_int, sm_flt, zero_mass);
      if (zero_mass) x = final_draw<T, 1>(z, pd, V, c, st.x, inv_sum(st.y), u, tot, sm_seg, sm_int, sm_flt, zero_mass);
    } else {
      const float u = philox_uniform(seed, req, (uint32_t)(L + 1), 3u);
      x = final_draw<T, 1>(z, nullptr, V, c, st.x, inv_sum(st.y), u, tot, sm_seg, sm_int, sm_flt, zero_mass);
    }
  }
  if (tid == 0) {
    out_tok[(size_t)r * (G + 1) + m] = x;
    n_accept[r] = m;
    n_out[r] = m + 1;
  }
}

template <typename T>
static cudaError_t launch_verify_t(const dspark_verify_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s) {
  const int B = a.dims.B, G = a.dims.gamma, V = a.dims.V;
  float4* rs = reinterpret_cast<float4*>(ws + L.vrs);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const T* tg = static_cast<const T*>(a.target_logits);
  k_verify_rowstats<T><<<dim3(B, G + 1, RS_PARTS), RS_THREADS, 0, s>>>(tg, a.offsets, a.ell, a.temp, V, rs);
  k_verify_finish<T><<<B, FIN_THREADS, 0, s>>>(tg, a.offsets, a.ell, a.tokens, a.pd_rows, a.pd_tok, a.temp,
                                               a.req_id, a.seed, G, V, rs, a.n_accept, a.out_tok, a.n_out, hdr);
  count_launches(2);
  return cudaGetLastError();
}

cudaError_t launch_verify(const dspark_verify_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s) {
  if (a.dims.dtype == DSPARK_BF16) return launch_verify_t<__nv_bfloat16>(a, ws, L, s);
  return launch_verify_t<float>(a, ws, L, s);
}

}  // namespace dspark
