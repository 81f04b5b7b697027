// Markov-head draft sampler: CUDA-core path and the per-row selection kernels.
//
// [DSpark] 方法细节, "序列阶段的依赖注入" / "马尔可夫头（Markov head）的实现":
// for k = 1..gamma, l_k = U_k + W1[x_{k-1}] W2, p_d^k = softmax(l_k / T), x_k ~ p_d^k.
// [DSpark] 方法细节, "置信度头的设计": c_k = sigmoid(w_h . h_k + w_e . W1[x_{k-1}]).
//
// One position k runs as
//   logits pass 1  per (row, vocabulary tile): max and sum of 2^(l c), argmax of l
//   k_select       per row: combine the tile partials, draw u, locate the tile
//                  that holds the draw, recompute that one tile, pick x_k; then
//                  copy W1[x_k] into the other E buffer and compute the
//                  confidence of position k + 1 (k_embed does position 1)
//   logits pass 2  recompute l, write p_d = 2^(l c - m) / S and p_d(x_k)
// The logits are recomputed rather than stored: storing them would cost a
// 4-byte write plus a 4-byte read per element, recomputing costs a 2-byte
// re-read of U (W2 stays in L2).  Every kernel evaluates l, l/T and exp(l/T - m)
// with the same helper functions, so the two logits passes of a path produce
// bit-identical values.  On the CUDA-core path the one tile k_select recomputes
// is bit-identical too (same FMA chain); on the tensor-core path (draft_tc.cu)
// k_select's CUDA-core recompute of that tile differs from the tensor-core sum
// only by fp32 rounding order (relative 1e-7), far inside the sampling margin.
#include <float.h>

#include <mutex>
#include <string>
#include <cstdlib>
#include <type_traits>
#include "common.cuh"
#include "draft_arith.cuh"
#include "internal.h"

namespace dspark {

// ---------------------------------------------------------------------------
// zh[b, k] = w_h . h[b, k, :]   (independent of the tokens: once per step)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) k_conf_hidden(const T* __restrict__ h, const T* __restrict__ w,
                                                     float* __restrict__ zh, int BG, int H) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= BG) return;
  float acc = 0.f;
  if (H > 0) {
    const T* hp = h + (size_t)warp * H;
    if ((H & 7) == 0) {
      // NU row loads of 16 (bf16) or 32 (fp32) bytes per lane in flight before
      // the first fma: one warp per row keeps too few bytes in flight otherwise.
      // The products are still added in increasing i.
      constexpr int NU = sizeof(T) == 2 ? 8 : 4;
      for (int i0 = lane * 8; i0 < H; i0 += 256 * NU) {
        float hv[NU][8];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          if (i0 + 256 * u < H) {
            load8_stream(hp + i0 + 256 * u, hv[u]);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) hv[u][e] = 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          if (i0 + 256 * u < H) {
            float wv[8];
            load8(w + i0 + 256 * u, wv);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(hv[u][e], wv[e], acc);
          }
        }
      }
    } else {
      for (int i = lane; i < H; i += 32) acc = fmaf(to_f32(hp[i]), to_f32(w[i]), acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) zh[warp] = acc;
}

// ---------------------------------------------------------------------------
// E[b] = W1[x_{k-1}], z_k = zh + w_e . E[b], c_k = sigmoid(z_k).  One warp per row.
// ---------------------------------------------------------------------------
// The row copy is skipped when E is null (the RNN head computes its own rows).
template <typename T, typename TE>
__device__ __forceinline__ void store_e(TE* dst, T v) {
  if constexpr (std::is_same<T, TE>::value)
    *dst = v;
  else
    *dst = to_f32(v);
}

template <typename T, typename TE>
__global__ void __launch_bounds__(256) k_embed(const int32_t* __restrict__ anchor, const int32_t* __restrict__ tokens,
                                               int k, const T* __restrict__ W1, const T* __restrict__ w,
                                               const float* __restrict__ zh, TE* __restrict__ E,
                                               float* __restrict__ conf_logit, float* __restrict__ conf, int B, int G,
                                               int V, int r, int H, WsHeader* hdr) {
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  int x = (k == 0) ? anchor[b] : tokens[(size_t)b * G + k - 1];
  if (x < 0 || x >= V) {
    if (lane == 0) report_error(hdr, DSPARK_BAD_INPUT, x);
    x = 0;
  }
  float acc = 0.f;
  if (r > 0) {
    const T* row = W1 + (size_t)x * r;
    const T* we = w + H;
    for (int i = lane; i < r; i += 32) {
      const T v = row[i];
      if (E) store_e(E + (size_t)b * r + i, v);
      acc = fmaf(to_f32(we[i]), to_f32(v), acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) {
    const float z = zh[(size_t)b * G + k] + acc;
    conf_logit[(size_t)b * G + k] = z;
    conf[(size_t)b * G + k] = 1.f / (1.f + expf(-z));
  }
}

// ---------------------------------------------------------------------------
// CUDA-core logits pass: a CTA owns CC_ROWS rows x CC_TW vocabulary columns, one
// column per thread.  The bias is a sequential FMA chain over the rank (the same
// chain k_select uses to recompute a tile).
// ---------------------------------------------------------------------------
constexpr int CC_ROWS = 16;
constexpr int CC_TW = 256;

template <typename T, typename TE, bool WRITE>
__global__ void __launch_bounds__(CC_TW) k_logits_cc(const T* __restrict__ U, const TE* __restrict__ E,
                                                     const T* __restrict__ W2, const float* __restrict__ temp,
                                                     int B, int G, int V, int r, int k, int ntiles,
                                                     float4* __restrict__ part, const float2* __restrict__ rowstat,
                                                     const int32_t* __restrict__ tokens, float* __restrict__ pd_rows,
                                                     float* __restrict__ pd_tok) {
  extern __shared__ float Es[];  // [CC_ROWS][r rounded up to 4]
  __shared__ float red_a[CC_TW / 32][CC_ROWS];
  __shared__ float red_b[CC_TW / 32][CC_ROWS];
  __shared__ int red_i[CC_TW / 32][CC_ROWS];
  __shared__ float row_m[CC_ROWS];
  __shared__ float row_invT[CC_ROWS];
  __shared__ int row_sampled[CC_ROWS];

  const int tile = blockIdx.x;
  const int b0 = blockIdx.y * CC_ROWS;
  const int nrows = min(CC_ROWS, B - b0);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int col = tile * CC_TW + tid;
  const bool valid = col < V;

  // rows padded to a multiple of 4 floats, so that the loop below reads four
  // rank entries of a row with one 16-byte shared-memory load
  const int rs = (r + 3) & ~3;
  for (int idx = tid; idx < CC_ROWS * rs; idx += CC_TW) {
    const int i = idx / rs, kk = idx - i * rs;
    Es[idx] = (i < nrows && kk < r) ? to_f32(E[(size_t)(b0 + i) * r + kk]) : 0.f;
  }
  if (tid < CC_ROWS) {
    const float T_ = (tid < nrows) ? temp[b0 + tid] : 1.f;
    row_sampled[tid] = T_ > 0.f;
    row_invT[tid] = row_scale(T_);
  }
  __syncthreads();

  float l[CC_ROWS];
#pragma unroll
  for (int i = 0; i < CC_ROWS; ++i) l[i] = 0.f;
  if (valid) {
    // each l[i] is one fma chain over the rank in ascending order (k_select
    // recomputes a tile with the same chain); four rank steps per shared-memory
    // load keep the loop on the FMA pipe
    const int r4 = r & ~3;
    for (int kk = 0; kk < r4; kk += 4) {
      const float w0 = ldf(W2 + (size_t)kk * V + col), w1 = ldf(W2 + (size_t)(kk + 1) * V + col);
      const float w2 = ldf(W2 + (size_t)(kk + 2) * V + col), w3 = ldf(W2 + (size_t)(kk + 3) * V + col);
#pragma unroll
      for (int i = 0; i < CC_ROWS; ++i) {
        const float4 e = *reinterpret_cast<const float4*>(&Es[i * rs + kk]);
        l[i] = fmaf(e.x, w0, l[i]);
        l[i] = fmaf(e.y, w1, l[i]);
        l[i] = fmaf(e.z, w2, l[i]);
        l[i] = fmaf(e.w, w3, l[i]);
      }
    }
    for (int kk = r4; kk < r; ++kk) {
      const float wv = ldf(W2 + (size_t)kk * V + col);
#pragma unroll
      for (int i = 0; i < CC_ROWS; ++i) l[i] = fmaf(Es[i * rs + kk], wv, l[i]);
    }
#pragma unroll
    for (int i = 0; i < CC_ROWS; ++i)
      if (i < nrows) l[i] = add_base(ldf(U + ((size_t)(b0 + i) * G + k) * V + col), l[i]);
  }

  if (!WRITE) {
    // ---- pass 1: per-row tile max of y = l/T, sum-exp, argmax of l ----
    float y[CC_ROWS];
#pragma unroll
    for (int i = 0; i < CC_ROWS; ++i) {
      y[i] = valid ? scale_logit(l[i], row_invT[i]) : -INFINITY;
      float mv = warp_max(y[i]);
      float av = valid ? l[i] : -INFINITY;
      int ai = valid ? col : INT_MAX;
      warp_argmax(av, ai);
      if (lane == 0) {
        red_a[wid][i] = mv;
        red_b[wid][i] = av;
        red_i[wid][i] = ai;
      }
    }
    __syncthreads();
    if (tid < CC_ROWS) {
      float mv = red_a[0][tid], av = red_b[0][tid];
      int ai = red_i[0][tid];
      for (int w_ = 1; w_ < CC_TW / 32; ++w_) {
        mv = fmaxf(mv, red_a[w_][tid]);
        argmax_merge(av, ai, red_b[w_][tid], red_i[w_][tid]);
      }
      row_m[tid] = mv;
      red_b[0][tid] = av;
      red_i[0][tid] = ai;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < CC_ROWS; ++i) {
      const float e = valid ? exp_shifted(y[i], row_m[i]) : 0.f;
      const float sv = warp_sum(e);
      if (lane == 0) red_a[wid][i] = sv;
    }
    __syncthreads();
    if (tid < nrows) {
      float sv = 0.f;
      for (int w_ = 0; w_ < CC_TW / 32; ++w_) sv += red_a[w_][tid];
      part[(size_t)(b0 + tid) * ntiles + tile] =
          make_float4(row_m[tid], sv, red_b[0][tid], __int_as_float(red_i[0][tid]));
    }
  } else {
    // ---- pass 2: p_d = exp(l/T - m) / S, one-hot for greedy rows ----
    if (!valid) return;
#pragma unroll
    for (int i = 0; i < CC_ROWS; ++i) {
      if (i >= nrows) break;
      const int b = b0 + i;
      const int x = tokens[(size_t)b * G + k];
      float p;
      if (row_sampled[i]) {
        const float2 st = rowstat[b];
        p = prob_from(scale_logit(l[i], row_invT[i]), st.x, inv_sum(st.y));
      } else {
        p = (col == x) ? 1.f : 0.f;
      }
      __stcs(pd_rows + ((size_t)b * G + k) * V + col, p);
      if (col == x) pd_tok[(size_t)b * G + k] = p;
    }
  }
}

// ---------------------------------------------------------------------------
// Per-row selection.  Partials part[b, t] = (m_t, s_t, argmax value, argmax idx)
// over tiles of `tw` columns.  Greedy rows take the global argmax.  Sampled
// rows: m = max m_t; tile masses q_t = s_t exp(m_t - m) summed in tile order
// give S and the prefix; target = u S; the tile where the prefix first exceeds
// the target is recomputed column by column with the pass-1 arithmetic and
// scanned in token order.
// ---------------------------------------------------------------------------
constexpr int SEL_THREADS = 256;

__device__ __forceinline__ float block_excl_scan_256(float v, float* sm, float& total) {
  // sm: >= 8 floats
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const float incl = warp_inclusive_scan(v);
  if (lane == 31) sm[wid] = incl;
  __syncthreads();
  float wpre = 0.f, tot = 0.f;
  for (int i = 0; i < SEL_THREADS / 32; ++i) {
    if (i < wid) wpre += sm[i];
    tot += sm[i];
  }
  __syncthreads();
  total = tot;
  return wpre + incl - v;
}

// After x_k is chosen the same CTA prepares position k + 1: it copies
// W1[x_k] into the other E buffer and evaluates that position's confidence,
// z_{k+1} = zh + w_e . W1[x_k] (the arithmetic of k_embed).
template <typename T, typename TE>
__device__ __forceinline__ void embed_next(int x, int b, int k, const T* __restrict__ W1, const T* __restrict__ w,
                                           const float* __restrict__ zh, TE* __restrict__ Enext,
                                           float* __restrict__ conf_logit, float* __restrict__ conf, int G, int r,
                                           int H) {
  if (k + 1 >= G || threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float acc = 0.f;
  if (r > 0) {
    const T* row = W1 + (size_t)x * r;
    const T* we = w + H;
    for (int i = lane; i < r; i += 32) {
      const T v = row[i];
      if (Enext) store_e(Enext + (size_t)b * r + i, v);
      acc = fmaf(to_f32(we[i]), to_f32(v), acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) {
    const float z = zh[(size_t)b * G + k + 1] + acc;
    conf_logit[(size_t)b * G + k + 1] = z;
    conf[(size_t)b * G + k + 1] = 1.f / (1.f + expf(-z));
  }
}

// Bytes of shared memory k_select stages a W2 tile chunk in.
constexpr int kSelStageBytes = 32768;

template <typename T, typename TE>
__global__ void __launch_bounds__(SEL_THREADS) k_select(const float4* __restrict__ part, int ntiles, int tw,
                                                        const T* __restrict__ U, const TE* __restrict__ Ecur,
                                                        const T* __restrict__ W2, const T* __restrict__ W1,
                                                        const T* __restrict__ w, const float* __restrict__ zh,
                                                        TE* __restrict__ Enext, const float* __restrict__ temp,
                                                        const uint32_t* __restrict__ req_id, uint64_t seed, int B,
                                                        int G, int V, int r, int H, int k, int32_t* __restrict__ tokens,
                                                        float2* __restrict__ rowstat, float* __restrict__ conf_logit,
                                                        float* __restrict__ conf, float2* __restrict__ pd_stat) {
  extern __shared__ float Erow[];  // [r] floats, then a [rows x tw] W2 chunk of T
  T* Ws = reinterpret_cast<T*>(Erow + r);
  __shared__ float sm[32];
  __shared__ int s_int[5];
  __shared__ float s_flt[4];
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const float4* P = part + (size_t)b * ntiles;
  const float T_ = temp[b];
  const bool sampled = T_ > 0.f;

  if (!sampled) {
    __shared__ int sai[SEL_THREADS / 32];
    float av = -INFINITY;
    int ai = INT_MAX;
    for (int t = tid; t < ntiles; t += SEL_THREADS) argmax_merge(av, ai, P[t].z, __float_as_int(P[t].w));
    warp_argmax(av, ai);
    if (lane == 0) {
      sm[wid] = av;
      sai[wid] = ai;
    }
    __syncthreads();
    if (tid == 0) {
      float v = sm[0];
      int i = sai[0];
      for (int w_ = 1; w_ < SEL_THREADS / 32; ++w_) argmax_merge(v, i, sm[w_], sai[w_]);
      tokens[(size_t)b * G + k] = i;
      rowstat[b] = make_float2(0.f, 1.f);
      if (pd_stat) pd_stat[(size_t)b * G + k] = make_float2(0.f, 1.f);
      s_int[4] = i;
    }
    __syncthreads();
    embed_next(s_int[4], b, k, W1, w, zh, Enext, conf_logit, conf, G, r, H);
    return;
  }

  // row max
  float mx = -INFINITY;
  for (int t = tid; t < ntiles; t += SEL_THREADS) mx = fmaxf(mx, P[t].x);
  mx = warp_max(mx);
  if (lane == 0) sm[wid] = mx;
  __syncthreads();
  if (tid == 0) {
    float v = sm[0];
    for (int w_ = 1; w_ < SEL_THREADS / 32; ++w_) v = fmaxf(v, sm[w_]);
    s_flt[0] = v;
  }
  __syncthreads();
  const float m = s_flt[0];
  __syncthreads();

  // tile masses in tile order: each thread owns a contiguous block of tiles
  const int cpt = (ntiles + SEL_THREADS - 1) / SEL_THREADS;
  const int t_lo = min(tid * cpt, ntiles), t_hi = min(t_lo + cpt, ntiles);
  float loc = 0.f;
  for (int t = t_lo; t < t_hi; ++t) loc += tile_mass(P[t].x, P[t].y, m);
  float S;
  const float pre = block_excl_scan_256(loc, sm, S);
  const float u = philox_uniform(seed, req_id[b], (uint32_t)(k + 1), 0u);
  const float target = u * S;

  // first tile whose inclusive prefix exceeds the target; also the last tile with mass
  if (tid == 0) {
    s_int[0] = INT_MAX;
    s_int[1] = -1;
  }
  __syncthreads();
  {
    float run = pre;
    int found = INT_MAX, lastpos = -1;
    for (int t = t_lo; t < t_hi; ++t) {
      const float q = tile_mass(P[t].x, P[t].y, m);
      if (found == INT_MAX && run + q > target) found = t;
      if (q > 0.f) lastpos = t;
      run += q;
    }
    if (found != INT_MAX) atomicMin(&s_int[0], found);
    if (lastpos >= 0) atomicMax(&s_int[1], lastpos);
  }
  __syncthreads();
  const bool hit = s_int[0] != INT_MAX;
  // a row without any positive mass (non-finite logits) falls back to tile 0
  const int tstar = min(max(hit ? s_int[0] : s_int[1], 0), ntiles - 1);
  // prefix before tstar: the owner recomputes it
  if (tstar >= t_lo && tstar < t_hi) {
    float run = pre;
    for (int t = t_lo; t < tstar; ++t) run += tile_mass(P[t].x, P[t].y, m);
    s_flt[1] = run;
  }
  for (int i = tid; i < r; i += SEL_THREADS) Erow[i] = to_f32(Ecur[(size_t)b * r + i]);
  __syncthreads();
  const float base = s_flt[1];

  // Recompute the tile's columns (tw <= SEL_THREADS) with the same sequential
  // FMA chain as the CUDA-core logits pass.  The W2 columns are staged through
  // shared memory in chunks of rows so that all loads of a chunk are in flight
  // together.
  const float c = row_scale(T_);
  const int col0 = tstar * tw;
  const int col = col0 + tid;
  const int chunk = max(1, min(r, kSelStageBytes / (tw * (int)sizeof(T))));
  float acc = 0.f;
  for (int kk0 = 0; kk0 < r; kk0 += chunk) {
    const int nr = min(chunk, r - kk0);
    const int total = nr * tw;
    // 32 independent loads per thread are in flight before any is stored
    for (int base = 0; base < total; base += SEL_THREADS * 32) {
      T vals[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int idx = base + j * SEL_THREADS + tid;
        const int rr = idx / tw, cc = idx - rr * tw;
        vals[j] = (idx < total && col0 + cc < V) ? W2[(size_t)(kk0 + rr) * V + col0 + cc] : T(0.f);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int idx = base + j * SEL_THREADS + tid;
        if (idx < total) Ws[idx] = vals[j];
      }
    }
    __syncthreads();
    if (tid < tw && col < V)
      for (int rr = 0; rr < nr; ++rr) acc = fmaf(Erow[kk0 + rr], to_f32(Ws[rr * tw + tid]), acc);
    __syncthreads();
  }
  float wv = 0.f;
  if (tid < tw && col < V) {
    const float l = add_base(ldf(U + ((size_t)b * G + k) * V + col), acc);
    wv = exp_shifted(scale_logit(l, c), m);
  }
  float tile_tot;
  const float excl = block_excl_scan_256(wv, sm, tile_tot);
  if (tid == 0) {
    s_int[2] = INT_MAX;
    s_int[3] = -1;
  }
  __syncthreads();
  if (tid < tw && col < V) {
    if (hit && base + (excl + wv) > target) atomicMin(&s_int[2], col);
    if (wv > 0.f) atomicMax(&s_int[3], col);
  }
  __syncthreads();
  if (tid == 0) {
    int x = (s_int[2] != INT_MAX) ? s_int[2] : s_int[3];
    if (x < 0) x = min(tstar * tw, V - 1);  // only reachable with non-finite logits
    tokens[(size_t)b * G + k] = x;
    rowstat[b] = make_float2(m, S);
    if (pd_stat) pd_stat[(size_t)b * G + k] = make_float2(m, S);
    s_int[4] = x;
  }
  __syncthreads();
  embed_next(s_int[4], b, k, W1, w, zh, Enext, conf_logit, conf, G, r, H);
}

// ---------------------------------------------------------------------------
// Host launcher
// ---------------------------------------------------------------------------
// CUDA-core path, per position: logits pass 1, k_select, logits pass 2.  The
// rows of the bias product are W1 rows (copied by k_embed / k_select) or, for
// the RNN head, the rows k_rnn_step computes before each position.
template <typename T, typename TE>
static cudaError_t launch_cuda_core(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s) {
  const dspark_dims& d = a.dims;
  const int B = d.B, G = d.gamma, V = d.V, r = d.r, H = d.H;
  const bool rnn = a.head == DSPARK_HEAD_RNN;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  float* zh = reinterpret_cast<float*>(ws + L.zh);
  TE* E = reinterpret_cast<TE*>(ws + L.E);
  float* S = reinterpret_cast<float*>(ws + L.rnn_s);
  float4* part = reinterpret_cast<float4*>(ws + L.part);
  float2* rowstat = reinterpret_cast<float2*>(ws + L.rowstat);
  const T* U = static_cast<const T*>(a.U);
  const T* W1 = static_cast<const T*>(a.W1);
  const T* W2 = static_cast<const T*>(a.W2);
  const T* h = static_cast<const T*>(a.h);
  const T* w = static_cast<const T*>(a.w);
  const int BG = B * G;

  k_conf_hidden<T><<<(BG + 7) / 8, 256, 0, s>>>(h, w, zh, BG, H);
  // position 1's confidence (and, for the Markov head, its W1 rows); later
  // positions are prepared by k_select
  k_embed<T, TE><<<(B + 7) / 8, 256, 0, s>>>(a.anchor, a.tokens, 0, W1, w, zh, rnn ? nullptr : E, a.conf_logit,
                                               a.conf, B, G, V, r, H, hdr);
  count_launches(2 + 3 * G);
  float* P = reinterpret_cast<float*>(ws + L.rnn_p);
  if (rnn) {
    const cudaError_t e = launch_rnn_hproj(a, P, reinterpret_cast<WsHeader*>(ws), s);
    if (e != cudaSuccess) return e;
  }
  const int tw = CC_TW;
  const int ntiles = (V + tw - 1) / tw;
  const size_t es_bytes = (size_t)CC_ROWS * ((r + 3) & ~3) * sizeof(float);
  if (es_bytes > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_logits_cc<T, TE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)es_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_logits_cc<T, TE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)es_bytes);
    if (e != cudaSuccess) return e;
  }
  const size_t sel_smem = (size_t)r * sizeof(float) + kSelStageBytes;
  const dim3 grid_cc(ntiles, (B + CC_ROWS - 1) / CC_ROWS);
  for (int k = 0; k < G; ++k) {
    // E holds two buffers: the rows of position k are in buffer k % 2
    TE* Ecur = E + (size_t)(k & 1) * B * r;
    TE* Enext = E + (size_t)((k + 1) & 1) * B * r;
    if (rnn) {
      // position k + 1 (1-based): s_k from s_{k-1}, e_{k+1} into Ecur
      const cudaError_t e = launch_rnn_step(a, k + 1, P, S + (size_t)(k & 1) * B * r,
                                            S + (size_t)((k + 1) & 1) * B * r, Ecur, s);
      if (e != cudaSuccess) return e;
    }
    k_logits_cc<T, TE, false><<<grid_cc, CC_TW, es_bytes, s>>>(U, Ecur, W2, a.temp, B, G, V, r, k, ntiles, part,
                                                                rowstat, a.tokens, a.pd_rows, a.pd_tok);
    k_select<T, TE><<<B, SEL_THREADS, sel_smem, s>>>(part, ntiles, tw, U, Ecur, W2, W1, w, zh, rnn ? nullptr : Enext,
                                                     a.temp, a.req_id, a.seed, B, G, V, r, H, k, a.tokens, rowstat,
                                                     a.conf_logit, a.conf, reinterpret_cast<float2*>(a.pd_stat));
    k_logits_cc<T, TE, true><<<grid_cc, CC_TW, es_bytes, s>>>(U, Ecur, W2, a.temp, B, G, V, r, k, ntiles, part,
                                                               rowstat, a.tokens, a.pd_rows, a.pd_tok);
  }
  return cudaGetLastError();
}

// The fused-sweep kernel serves the tensor-core shapes unless
// DSPARK_DRAFT_LAUNCH=two_pass or per_pass selects the pass kernels;
// DSPARK_DRAFT_LAUNCH=fused takes it for the RNN head at every batch.
static int draft_launch_mode() {  // 0: pass kernels, 1: default, 2: fused always
  static int mode = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* e = getenv("DSPARK_DRAFT_LAUNCH");
    const std::string v = e ? e : "";
    mode = (v == "per_pass" || v == "two_pass") ? 0 : (v == "fused" ? 2 : 1);
  });
  return mode;
}
static bool fused_launch_enabled() { return draft_launch_mode() != 0; }

// The RNN head above this batch runs the pass kernels with the recurrent step
// on the tensor cores: measured at r256 gamma 7, the fused form's recurrent
// units (fp32, one CTA's share at a time) cost more there (B1024: 2.70 against
// 2.46 ms; B256: 0.84 against 0.90 ms).
constexpr int kRnnFusedMaxB = 512;

// The RNN head's recurrent step on the tensor cores (bf16 tensor-core shapes)
// unless DSPARK_RNN_STEP=cuda_core keeps k_rnn_step.
static bool rnn_step_tc_enabled() {
  static int tc = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* e = getenv("DSPARK_RNN_STEP");
    tc = (e && std::string(e) == "cuda_core") ? 0 : 1;
  });
  return tc != 0;
}

template <typename T>
static cudaError_t launch_draft_t(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s,
                                  DraftOverlap* ov) {
  const dspark_dims& d = a.dims;
  // without p_d rows: the fused-sweep kernel only (its select yields p_d(x) and (m, S))
  if (!a.pd_rows) return draft_tc_supported(d) ? launch_draft_fused(a, ws, L, s, ov) : cudaErrorNotSupported;
  if (a.head == DSPARK_HEAD_RNN) {
    if (!draft_tc_supported(d)) return launch_cuda_core<T, T>(a, ws, L, s);
    // the fused-sweep kernel (either form) with the recurrent step between
    // sweeps, up to kRnnFusedMaxB requests unless DSPARK_DRAFT_LAUNCH says otherwise
    if (draft_launch_mode() == 2 || (draft_launch_mode() == 1 && d.B <= kRnnFusedMaxB)) {
      const cudaError_t fe = launch_draft_fused(a, ws, L, s, ov);
      if (fe != cudaErrorNotSupported) return fe;
    }
    // tensor-core passes, one launch per pass; before each position the
    // recurrent step writes its rows (bf16) and k_embed its confidences
    const int B = d.B, r = d.r, BG = B * d.gamma;
    float* zh = reinterpret_cast<float*>(ws + L.zh);
    float* P = reinterpret_cast<float*>(ws + L.rnn_p);
    float* S = reinterpret_cast<float*>(ws + L.rnn_s);
    T* Erows = reinterpret_cast<T*>(ws + L.E);
    const T* W1 = static_cast<const T*>(a.W1);
    const T* w = static_cast<const T*>(a.w);
    k_conf_hidden<T><<<(BG + 7) / 8, 256, 0, s>>>(static_cast<const T*>(a.h), w, zh, BG, d.H);
    count_launches(1);
    cudaError_t e = launch_rnn_hproj(a, P, reinterpret_cast<WsHeader*>(ws), s);
    if (e != cudaSuccess) return e;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    // the recurrent step: on the tensor cores (z'' and the packed weights), or k_rnn_step
    const bool tc_step = std::is_same<T, __nv_bfloat16>::value && rnn_step_tc_enabled();
    auto* Z = reinterpret_cast<__nv_bfloat16*>(ws + L.rnn_z);
    auto* Wz = reinterpret_cast<__nv_bfloat16*>(ws + L.rnn_wz);
    float* pre = reinterpret_cast<float*>(ws + L.rnn_pre);
    if (tc_step && (e = launch_rnn_pack_wz(a, Wz, s)) != cudaSuccess) return e;
    const std::function<cudaError_t(int)> hook = [&](int k) {
      const float* s_prev = S + (size_t)(k & 1) * B * r;
      float* s_new = S + (size_t)((k + 1) & 1) * B * r;
      const cudaError_t e2 = tc_step ? launch_rnn_step_tc(a, k + 1, P, s_prev, s_new,
                                                          reinterpret_cast<__nv_bfloat16*>(Erows), Z, Wz, pre, hdr, s)
                                     : launch_rnn_step(a, k + 1, P, s_prev, s_new, Erows, s);
      if (e2 != cudaSuccess) return e2;
      k_embed<T, T><<<(B + 7) / 8, 256, 0, s>>>(a.anchor, a.tokens, k, W1, w, zh, nullptr, a.conf_logit, a.conf, B,
                                                d.gamma, d.V, r, d.H, hdr);
      count_launches(1);
      return cudaGetLastError();
    };
    return launch_draft_tc(a, ws, L, s, &hook, Erows);
  }
  if (draft_tc_supported(d)) {
    // tensor-core path: the fused-sweep persistent kernel (which forms w_h . h
    // itself), else the two-pass kernel (DSPARK_DRAFT_LAUNCH=two_pass or
    // per_pass selects the latter)
    if (fused_launch_enabled()) {
      const cudaError_t e = launch_draft_fused(a, ws, L, s, ov);
      if (e != cudaErrorNotSupported) return e;
    }
    const int BG = d.B * d.gamma;
    k_conf_hidden<T><<<(BG + 7) / 8, 256, 0, s>>>(static_cast<const T*>(a.h), static_cast<const T*>(a.w),
                                                  reinterpret_cast<float*>(ws + L.zh), BG, d.H);
    count_launches(1);
    return launch_draft_tc(a, ws, L, s);
  }
  return launch_cuda_core<T, T>(a, ws, L, s);
}

cudaError_t launch_draft(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s,
                         DraftOverlap* ov) {
  if (ov) ov->armed = false;
  if (a.dims.dtype == DSPARK_BF16) return launch_draft_t<__nv_bfloat16>(a, ws, L, s, ov);
  return launch_draft_t<float>(a, ws, L, s, ov);
}

}  // namespace dspark
