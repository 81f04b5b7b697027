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
// k_verify_final     one CTA per slice of a request's final row: the accept
//                    tests (one warp, p_t at each draft token from the row
//                    statistics), the first rejection m, then the weights of
//                    the final draw (residual max(0, p_t - p_d), or the bonus
//                    2^(y - max)) summed per 256-token chunk
// k_verify_pick      one warp per request: inverse CDF over the chunk sums in
//                    token order, then a re-read of the one chunk that holds
//                    the draw
#include <algorithm>

#include "common.cuh"
#include "draft_arith.cuh"
#include "internal.h"

namespace dspark {

constexpr int RS_THREADS = 256;
constexpr int RS_UNROLL = 2;            // 16-byte loads in flight per thread

// The temperature of every kept row (flattened row offsets[r] + j, j <= l_r),
// so that the row statistics need one load per row.
__global__ void k_verify_rowmap(const int32_t* __restrict__ offsets, const int32_t* __restrict__ ell,
                                const float* __restrict__ temp, int B, int G, float* __restrict__ rowT) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int r = idx / (G + 1), j = idx % (G + 1);
  if (r < B && j <= ell[r]) rowT[offsets[r] + j] = temp[r];
}

// Each kept row is split into RS_PARTS contiguous slices, one CTA per (row,
// slice) item of the N_v = offsets[B] kept rows (flattened row order, so that
// the CTAs past N_v, the grid's tail, return at once), RS_UNROLL 16-byte loads
// in flight per thread.  Partial per (row, slice): sampled rows store (max y,
// sum 2^(y - max)); greedy rows store (argmax value, argmax index).
template <typename T>
__global__ void __launch_bounds__(RS_THREADS) k_verify_rowstats(const T* __restrict__ target,
                                                                const int32_t* __restrict__ offsets,
                                                                const float* __restrict__ rowT, int B, int V,
                                                                float4* __restrict__ rsp) {
  __shared__ float sm_a[RS_THREADS / 32], sm_b[RS_THREADS / 32];
  __shared__ int sm_i[RS_THREADS / 32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int w = (int)blockIdx.x;
  if (w >= offsets[B] * RS_PARTS) return;
  const bool vec = (V & 7) == 0;
  const int span = ((V + RS_PARTS - 1) / RS_PARTS + 7) & ~7;  // multiple of 8: vector loads stay aligned
  {
    const int n = w / RS_PARTS, part = w % RS_PARTS;
    const float T_ = rowT[n];
    const T* z = target + (size_t)n * V;
    const bool sampled = T_ > 0.f;
    const float c = row_scale(T_);
    const int lo = min(part * span, V), hi = min(lo + span, V);
    float m = -INFINITY, s = 0.f, av = -INFINITY;
    int ai = INT_MAX;
    if (vec) {
      for (int i0 = lo + tid * 8; i0 < hi; i0 += RS_THREADS * 8 * RS_UNROLL) {
        float v[RS_UNROLL][8];
#pragma unroll
        for (int u = 0; u < RS_UNROLL; ++u)
          if (i0 + u * RS_THREADS * 8 < hi) load8_stream(z + i0 + u * RS_THREADS * 8, v[u]);
#pragma unroll
        for (int u = 0; u < RS_UNROLL; ++u) {
          if (i0 + u * RS_THREADS * 8 >= hi) break;
          if (sampled) {
            // c > 0: the max of z c is c times the max of z; each weight is
            // 2^(z c - m) with one rounding (fma)
            float zm = v[u][0];
#pragma unroll
            for (int q = 1; q < 8; ++q) zm = fmaxf(zm, v[u][q]);
            const float lm = scale_logit(zm, c);
            if (lm > m) {
              s = s * ex2_ftz(__fsub_rn(m, lm));
              m = lm;
            }
            const float nm = -m;
            float s2[2] = {0.f, 0.f};
#pragma unroll
            for (int q = 0; q < 8; ++q) s2[q & 1] += ex2_ftz(fmaf(v[u][q], c, nm));
            s += s2[0] + s2[1];
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) argmax_merge(av, ai, v[u][q], i0 + u * RS_THREADS * 8 + q);
          }
        }
      }
    } else {
      for (int i = lo + tid; i < hi; i += RS_THREADS) {
        const float y0 = to_f32(z[i]);
        if (sampled) {
          const float y = scale_logit(y0, c);
          if (y > m) {
            s = s * exp2f(m - y);
            m = y;
          }
          s += exp_shifted(y, m);
        } else {
          argmax_merge(av, ai, y0, i);
        }
      }
    }
    if (sampled) {
      warp_lse(m, s);
      if (lane == 0) {
        sm_a[wid] = m;
        sm_b[wid] = s;
      }
    } else {
      warp_argmax(av, ai);
      if (lane == 0) {
        sm_a[wid] = av;
        sm_i[wid] = ai;
      }
    }
    __syncthreads();
    if (tid == 0) {
      float4 out;
      if (sampled) {
        float M = sm_a[0], S = sm_b[0];
        for (int w_ = 1; w_ < RS_THREADS / 32; ++w_) lse_merge(M, S, sm_a[w_], sm_b[w_]);
        out = make_float4(M, S, 0.f, 0.f);
      } else {
        float A = sm_a[0];
        int I = sm_i[0];
        for (int w_ = 1; w_ < RS_THREADS / 32; ++w_) argmax_merge(A, I, sm_a[w_], sm_i[w_]);
        out = make_float4(A, __int_as_float(I), 0.f, 0.f);
      }
      rsp[(size_t)n * RS_PARTS + part] = out;
    }
  }
}

// q(v) of the final draw: residual max(0, p_t - p_d) or the bonus weight 2^(y - m)
template <typename T, int MODE>  // MODE 0: residual, 1: target weights
__device__ __forceinline__ float final_weight(const T* z, const float* pd, int v, float c, float m, float invS) {
  const float y = scale_logit(to_f32(z[v]), c);
  if (MODE == 1) return exp_shifted(y, m);
  return fmaxf(0.f, __fsub_rn(prob_from(y, m, invS), pd[v]));
}

// The final draw works on 256-token chunks (8 tokens per lane of a warp).
constexpr int FN_THREADS = 256;
constexpr int FN_SLICES = 8;        // CTAs per request's final row
constexpr int PK_WARPS = 4;         // requests per CTA of k_verify_pick
constexpr int AC_WARPS = 8;         // warps per request in k_verify_accept
constexpr int PK_REG = 24;          // chunk sums per lane the pick keeps in registers (V <= 196608)

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

// One CTA per request: warp w takes the rows j = w, w + AC_WARPS, .. <= L of
// the request; the row statistics come from its RS_PARTS slice partials (one
// per lane, merged across the warp); for j < L the accept test of position
// j + 1 (p_t at the draft token from the statistics, u * p_d < p_t, or the
// argmax compare at temperature 0).  The first rejection ends the accepted
// prefix: vm[r] = m, and the final row's record goes to fmeta / fstat.
template <typename T>
__global__ void __launch_bounds__(AC_WARPS * 32) k_verify_accept(const T* __restrict__ target,
                                                                 const int32_t* __restrict__ offsets,
                                                                 const int32_t* __restrict__ ell,
                                                                 const int32_t* __restrict__ tokens,
                                                                 const float* __restrict__ pd_tok,
                                                                 const float* __restrict__ temp,
                                                                 const uint32_t* __restrict__ req_id, uint64_t seed,
                                                                 int G, int V, const float4* __restrict__ rs,
                                                                 int32_t* __restrict__ vm, int4* __restrict__ fmeta,
                                                                 float4* __restrict__ fstat, WsHeader* hdr) {
  static_assert(RS_PARTS <= 32, "one slice partial per lane");
  __shared__ float4 s_st[DSPARK_MAX_GAMMA + 1];
  __shared__ unsigned s_rej[(DSPARK_MAX_GAMMA + 31) / 32 + 1];
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int L = ell[r];
  const float T_ = temp[r];
  const bool sampled = T_ > 0.f;
  const float c = row_scale(T_);
  const int base = offsets[r];
  if (threadIdx.x < (DSPARK_MAX_GAMMA + 31) / 32 + 1) s_rej[threadIdx.x] = 0u;
  __syncthreads();
  for (int j = wid; j <= L; j += AC_WARPS) {
    const size_t row = (size_t)base + j;
    const float4 p = lane < RS_PARTS ? rs[row * RS_PARTS + lane]
                                     : make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(INT_MAX));
    int x = 0;
    float ztok = 0.f;
    if (j < L) {
      x = tokens[(size_t)r * G + j];
      if (x < 0 || x >= V) {
        if (lane == 0) report_error(hdr, DSPARK_BAD_INPUT, x);
        x = 0;
      }
      if (sampled) ztok = to_f32(target[row * V + x]);  // the same address in every lane
    }
    float4 st;
    if (sampled) {
      float M = p.x, S = p.y;
      warp_lse(M, S);
      st = make_float4(M, S, 0.f, 0.f);
    } else {
      float av = p.x;
      int ai = __float_as_int(p.y);
      warp_argmax(av, ai);
      st = make_float4(0.f, 1.f, __int_as_float(ai), 0.f);
    }
    if (lane == 0) {
      s_st[j] = st;
      if (j < L) {
        bool acc;
        if (sampled) {
          const float ptok = prob_from(scale_logit(ztok, c), st.x, inv_sum(st.y));
          const float u = philox_uniform(seed, req_id[r], (uint32_t)(j + 1), 1u);
          acc = __fmul_rn(u, pd_tok[(size_t)r * G + j]) < ptok;
        } else {
          acc = x == __float_as_int(st.z);
        }
        if (!acc) atomicOr(&s_rej[j >> 5], 1u << (j & 31));
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = L;
    for (int q = 0; q * 32 < L; ++q)
      if (s_rej[q]) {
        m = q * 32 + __ffs(s_rej[q]) - 1;
        break;
      }
    vm[r] = m;
    const float4 st = s_st[m];
    // sampled: (max, 1/sum, scale); greedy: the argmax of the final row, the
    // output token
    fmeta[r] = make_int4(base + m, m < L ? 1 : 0, sampled ? 1 : 0, m);
    fstat[r] = sampled ? make_float4(st.x, inv_sum(st.y), c, 0.f) : make_float4(st.z, 0.f, 0.f, 0.f);
  }
}

// Chunk sums of the final draw's weights, one CTA per slice of a sampled
// request's final row (the accepted count and the row's statistics come from
// k_verify_accept): chunk c of request r goes to fin[r][(c % E) 32 + c / E]
// (E = ceil(nch / 32), the pick's lane-major order) as (mode weight, bonus
// weight): the mode weight is the residual for a rejecting row and the bonus
// weight otherwise; the bonus weight also serves a residual of zero mass.
template <typename T>
__global__ void __launch_bounds__(FN_THREADS) k_verify_final(const T* __restrict__ target,
                                                             const float* __restrict__ pd_rows, int G, int V,
                                                             const int4* __restrict__ fmeta,
                                                             const float4* __restrict__ fstat,
                                                             float2* __restrict__ fin, bool row_free) {
  const int r = blockIdx.x, slice = blockIdx.y;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int4 fm = fmeta[r];
  if (!fm.z) return;  // greedy: no draw
  const float4 fs = fstat[r];
  // without p_d rows the residual is drawn by rejection from p_t: p_t's weights only
  const bool resid = fm.y != 0 && !row_free;
  const int m = fm.w;
  const float M = fs.x, invS = fs.y, c = fs.z;
  const T* z = target + (size_t)fm.x * V;
  const float* pd = resid ? pd_rows + ((size_t)r * G + m) * V : nullptr;
  const bool vec = (V & 7) == 0;
  const int nch = (V + 255) >> 8, E = (nch + 31) >> 5;
  const int cps = (nch + FN_SLICES - 1) / FN_SLICES;
  const int c_lo = slice * cps, c_hi = min(c_lo + cps, nch);
  float2* F = fin + (size_t)r * E * 32;
#pragma unroll 2
  for (int ch = c_lo + wid; ch < c_hi; ch += FN_THREADS / 32) {
    const int v0 = ch * 256 + lane * 8;
    float qb[8], qm[8];
    if (resid) {
      // one read of the chunk: e = 2^(y - max) is the bonus weight, e / S - p_d
      // the residual's
      if (vec && v0 + 8 <= V) {
        float zv[8], pv[8];
        load8_stream(z + v0, zv);
        load8_stream(pd + v0, pv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          qb[e] = exp_shifted(scale_logit(zv[e], c), M);
          qm[e] = fmaxf(0.f, __fsub_rn(__fmul_rn(qb[e], invS), pv[e]));
        }
      } else {
        chunk_weights<T, 1>(z, nullptr, v0, V, vec, c, M, invS, qb);
        chunk_weights<T, 0>(z, pd, v0, V, vec, c, M, invS, qm);
      }
    } else {
      chunk_weights<T, 1>(z, nullptr, v0, V, vec, c, M, invS, qb);
#pragma unroll
      for (int e = 0; e < 8; ++e) qm[e] = qb[e];
    }
    const float tm = warp_sum(lane_sum8(qm));
    const float tb = warp_sum(lane_sum8(qb));
    if (lane == 0) F[(ch % E) * 32 + ch / E] = make_float2(tm, tb);
  }
}

// One warp per request: the outputs, and for a sampled row the inverse-CDF
// draw over the final row in token order: lane l holds the chunk sums
// [l E, l E + E) (in registers up to PK_REG of them), a warp scan finds the
// lane, a scan of that lane's sums the chunk whose running sum first exceeds
// u * total, and a re-read of that chunk the token.  Rounding that leaves no
// crossing falls back to the last positive weight.  A residual of zero mass
// (reachable only through rounding) draws from p_t instead, with the same u.
// what the row-free (rejection) residual reads
struct RowFree {
  bool on;
  int r;
  const void* U;
  const void* W1;
  const void* W2;
  const int32_t* anchor;
  const float* pd_stat;
};

template <typename T>
__global__ void __launch_bounds__(PK_WARPS * 32) k_verify_pick(const T* __restrict__ target,
                                                               const int32_t* __restrict__ ell,
                                                               const int32_t* __restrict__ tokens,
                                                               const float* __restrict__ pd_rows,
                                                               const uint32_t* __restrict__ req_id, uint64_t seed,
                                                               int B, int G, int V, const int4* __restrict__ fmeta,
                                                               const float4* __restrict__ fstat,
                                                               const float2* __restrict__ fin,
                                                               int32_t* __restrict__ n_accept,
                                                               int32_t* __restrict__ out_tok,
                                                               int32_t* __restrict__ n_out,
                                                               const int32_t* __restrict__ commit_cap,
                                                               WsHeader* __restrict__ hdr, RowFree rf) {
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * PK_WARPS + (threadIdx.x >> 5);
  if (r >= B) return;
  const int nch = (V + 255) >> 8, E = (nch + 31) >> 5;
  const int c0 = lane * E;
  const float2* F = fin + (size_t)r * E * 32;
  // the chunk sums do not depend on the record: their loads go out with it
  float2 f[PK_REG];
  if (E <= PK_REG) {
#pragma unroll
    for (int t = 0; t < PK_REG; ++t) {
      if (t >= E) break;
      f[t] = c0 + t < nch ? F[t * 32 + lane] : make_float2(0.f, 0.f);
    }
  }
  const int4 fm = fmeta[r];
  const float4 fs = fstat[r];
  const int m = fm.w, L = ell[r];
  // cap-accept: commit the first min(m, window) + 1 emitted tokens; past the
  // window the last committed token is the accepted draft token
  int nout = m + 1;
  if (commit_cap) {
    int c = commit_cap[r];
    if (c < 0 || c > G) {
      if (lane == 0) report_error(hdr, DSPARK_BAD_INPUT, r);
      c = c < 0 ? 0 : G;
    }
    nout = min(m, c) + 1;
  }
  for (int i = lane; i <= G; i += 32)
    out_tok[(size_t)r * (G + 1) + i] = (i < m && i < nout) ? tokens[(size_t)r * G + i] : -1;
  int x;
  if (!fm.z) {
    x = __float_as_int(fs.x);
  } else {
    const bool resid = fm.y != 0;
    const bool rejection = resid && rf.on;  // residual by rejection from p_t
    auto entry = [&](int t) { return E <= PK_REG ? f[t] : F[t * 32 + lane]; };
    // lane sums of its chunks (both kinds of weight), and its last chunk with
    // positive weight of each kind
    float sm = 0.f, sb = 0.f;
    int lm = -1, lb = -1;
#pragma unroll
    for (int t = 0; t < PK_REG; ++t) {
      if (t >= E || c0 + t >= nch) break;
      const float2 e = entry(t);
      sm = __fadd_rn(sm, e.x);
      sb = __fadd_rn(sb, e.y);
      if (e.x > 0.f) lm = c0 + t;
      if (e.y > 0.f) lb = c0 + t;
    }
    for (int t = PK_REG; t < E; ++t) {  // beyond the register window
      if (c0 + t >= nch) break;
      const float2 e = F[t * 32 + lane];
      sm = __fadd_rn(sm, e.x);
      sb = __fadd_rn(sb, e.y);
      if (e.x > 0.f) lm = c0 + t;
      if (e.y > 0.f) lb = c0 + t;
    }
    const float tot_m = warp_sum(sm);
    const T* zrow = target + (size_t)fm.x * V;
    const float M = fs.x, invS = fs.y, c = fs.z;
    // inverse-CDF draw with u over the chunk sums (use_b: p_t's weights, else the
    // mode's), then the token by a re-read of the crossing chunk
    auto draw = [&](float u, bool use_b) -> int {
      int x = -1;
      const float sl = use_b ? sb : sm;
      const float incl = warp_inclusive_scan(sl);
      const float total = __shfl_sync(FULL, incl, 31);
      const float tgt = u * total;
      float ex = __shfl_up_sync(FULL, incl, 1);
      if (lane == 0) ex = 0.f;
      const unsigned over = __ballot_sync(FULL, total > 0.f && incl > tgt);
      // the crossing lane walks its own chunks
      int cstar = -1, clast = -1;
      float cpre = 0.f, run = ex;
#pragma unroll
      for (int t = 0; t < PK_REG; ++t) {
        if (t >= E || c0 + t >= nch) break;
        const float2 e = entry(t);
        const float w = use_b ? e.y : e.x;
        const float nr = __fadd_rn(run, w);
        if (w > 0.f) clast = c0 + t;
        if (cstar < 0 && nr > tgt) {
          cstar = c0 + t;
          cpre = run;
        }
        run = nr;
      }
      for (int t = PK_REG; t < E; ++t) {
        if (c0 + t >= nch) break;
        const float2 e = F[t * 32 + lane];
        const float w = use_b ? e.y : e.x;
        const float nr = __fadd_rn(run, w);
        if (w > 0.f) clast = c0 + t;
        if (cstar < 0 && nr > tgt) {
          cstar = c0 + t;
          cpre = run;
        }
        run = nr;
      }
      bool in_chunk = false;
      if (over) {
        const int Lw = __ffs(over) - 1;
        in_chunk = __shfl_sync(FULL, cstar >= 0 ? 1 : 0, Lw) != 0;
        const int cs = __shfl_sync(FULL, cstar, Lw), cl = __shfl_sync(FULL, clast, Lw);
        cpre = __shfl_sync(FULL, cpre, Lw);
        cstar = in_chunk ? cs : cl;
      } else {
        cstar = -1;
      }
      if (cstar < 0) {
        // no crossing: the last chunk with positive weight
        int lc = use_b ? lb : lm;
        for (int o = 16; o > 0; o >>= 1) lc = max(lc, __shfl_xor_sync(FULL, lc, o));
        cstar = lc;
        in_chunk = false;
      }
      if (cstar >= 0) {
        const T* z = zrow;
        const float* pd = (resid && !rf.on) ? pd_rows + ((size_t)r * G + m) * V : nullptr;
        const bool vec = (V & 7) == 0;
        const int v0 = cstar * 256 + lane * 8;
        float q[8];
        if (resid && !use_b && !rf.on)
          chunk_weights<T, 0>(z, pd, v0, V, vec, c, M, invS, q);
        else
          chunk_weights<T, 1>(z, nullptr, v0, V, vec, c, M, invS, q);
        const float ls = lane_sum8(q);
        const float li = warp_inclusive_scan(ls);
        int lastp = -1;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (q[e] > 0.f) lastp = v0 + e;
        if (in_chunk) {
          const unsigned ov = __ballot_sync(FULL, cpre + li > tgt);
          if (ov) {
            const int Ll = __ffs(ov) - 1;
            float pre = __shfl_up_sync(FULL, li, 1);
            pre = __shfl_sync(FULL, (lane == 0) ? 0.f : pre, Ll);
            int xl = -1;
            if (lane == Ll) {
              float acc = cpre + pre;
              for (int e = 0; e < 8; ++e) {
                acc += q[e];
                if (acc > tgt) {
                  xl = v0 + e;
                  break;
                }
              }
              if (xl < 0) xl = lastp;
            }
            x = __shfl_sync(FULL, xl, Ll);
          }
        }
        if (x < 0) {  // rounding left no crossing: last positive weight of the chunk
          int lp = lastp;
          for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(FULL, lp, o));
          x = lp;
        }
      }
      return x;
    };
    if (!rejection) {
      const float u = resid ? philox_uniform(seed, req_id[r], (uint32_t)(m + 1), 2u)
                            : philox_uniform(seed, req_id[r], (uint32_t)(L + 1), 3u);
      x = draw(u, resid && !(tot_m > 0.f));
    } else {
      // proposals v ~ p_t, accepted iff u p_t(v) < p_t(v) - p_d(v); p_d(v) of the
      // Markov head recomputed at v from U, W1[x_m] and the row's (max, sum)
      const int xp0 = (m == 0) ? rf.anchor[r] : tokens[(size_t)r * G + m - 1];
      const int xp = (xp0 >= 0 && xp0 < V) ? xp0 : 0;
      const float2 st = reinterpret_cast<const float2*>(rf.pd_stat)[(size_t)r * G + m];
      const float dinv = inv_sum(st.y);
      const T* W1r = static_cast<const T*>(rf.W1) + (size_t)xp * rf.r;
      const T* W2 = static_cast<const T*>(rf.W2);
      const T* Ur = static_cast<const T*>(rf.U) + ((size_t)r * G + m) * V;
      auto pd_at = [&](int v) -> float {  // warp-wide, the same value in every lane
        float acc = 0.f;
        for (int i = lane; i < rf.r; i += 32) acc = fmaf(to_f32(W1r[i]), to_f32(W2[(size_t)i * V + v]), acc);
        acc = warp_sum(acc);
        return prob_from(scale_logit(add_base(to_f32(Ur[v]), acc), c), st.x, dinv);
      };
      const uint32_t req = req_id[r];
      x = -1;
      for (int t = 0; t < DSPARK_RESIDUAL_TRIALS && x < 0; ++t) {
        const int v = max(draw(philox_uniform(seed, req, (uint32_t)(m + 1), 2u, (uint32_t)t), false), 0);
        const float pt = prob_from(scale_logit(to_f32(zrow[v]), c), M, invS);
        const float pdv = pd_at(v);
        const float w = philox_uniform(seed, req, (uint32_t)(m + 1), 4u, (uint32_t)t);
        if (__fmul_rn(w, pt) < __fsub_rn(pt, pdv)) x = v;
      }
      if (x < 0) {
        // no proposal accepted: the residual by inverse CDF, recomputing p_d at
        // every token (two passes over the vocabulary; one lane per token)
        const float u = philox_uniform(seed, req, (uint32_t)(m + 1), 2u, (uint32_t)DSPARK_RESIDUAL_TRIALS);
        auto q_at = [&](int v) -> float {
          if (v >= V) return 0.f;
          float acc = 0.f;
          for (int i = 0; i < rf.r; ++i) acc = fmaf(to_f32(W1r[i]), to_f32(W2[(size_t)i * V + v]), acc);
          const float pdv = prob_from(scale_logit(add_base(to_f32(Ur[v]), acc), c), st.x, dinv);
          return fmaxf(0.f, __fsub_rn(prob_from(scale_logit(to_f32(zrow[v]), c), M, invS), pdv));
        };
        float Q = 0.f;
        for (int v0 = 0; v0 < V; v0 += 32) Q = __fadd_rn(Q, warp_sum(q_at(v0 + lane)));
        if (!(Q > 0.f)) {
          x = draw(u, false);  // zero residual mass: p_t
        } else {
          const float tgt = u * Q;
          float run = 0.f;
          int lastp = -1;
          for (int v0 = 0; v0 < V && x < 0; v0 += 32) {
            const float q = q_at(v0 + lane);
            const float incl = __fadd_rn(run, warp_inclusive_scan(q));
            const unsigned ov = __ballot_sync(FULL, incl > tgt);
            const unsigned pos = __ballot_sync(FULL, q > 0.f);
            if (pos) lastp = v0 + 31 - __clz(pos);
            if (ov) x = v0 + __ffs(ov) - 1;
            run = __shfl_sync(FULL, incl, 31);
          }
          if (x < 0) x = lastp;
        }
      }
    }
  }
  if (lane == 0) {
    if (nout == m + 1) out_tok[(size_t)r * (G + 1) + m] = x;
    n_accept[r] = m;
    n_out[r] = nout;
  }
}

template <typename T>
static cudaError_t launch_verify_t(const dspark_verify_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s) {
  const int B = a.dims.B, G = a.dims.gamma, V = a.dims.V;
  if (B == 0) return cudaSuccess;
  float4* rs = reinterpret_cast<float4*>(ws + L.vrs);
  float2* fin = reinterpret_cast<float2*>(ws + L.vfin);
  int32_t* vm = reinterpret_cast<int32_t*>(ws + L.vm);
  float* rowT = reinterpret_cast<float*>(ws + L.vrowT);
  int4* fmeta = reinterpret_cast<int4*>(ws + L.vfmeta);
  float4* fstat = reinterpret_cast<float4*>(ws + L.vfstat);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const T* tg = static_cast<const T*>(a.target_logits);
  const int nw = (B + PK_WARPS - 1) / PK_WARPS;
  k_verify_rowmap<<<(B * (G + 1) + 255) / 256, 256, 0, s>>>(a.offsets, a.ell, a.temp, B, G, rowT);
  k_verify_rowstats<T><<<B * (G + 1) * RS_PARTS, RS_THREADS, 0, s>>>(tg, a.offsets, rowT, B, V, rs);
  k_verify_accept<T><<<B, AC_WARPS * 32, 0, s>>>(tg, a.offsets, a.ell, a.tokens, a.pd_tok, a.temp, a.req_id,
                                                  a.seed, G, V, rs, vm, fmeta, fstat, hdr);
  const bool row_free = a.residual_mode == DSPARK_RESIDUAL_REJECTION;
  const RowFree rf{row_free, a.dims.r, a.U, a.W1, a.W2, a.anchor, a.pd_stat};
  k_verify_final<T><<<dim3(B, FN_SLICES), FN_THREADS, 0, s>>>(tg, a.pd_rows, G, V, fmeta, fstat, fin, row_free);
  k_verify_pick<T><<<nw, PK_WARPS * 32, 0, s>>>(tg, a.ell, a.tokens, a.pd_rows, a.req_id, a.seed, B, G, V, fmeta,
                                                fstat, fin, a.n_accept, a.out_tok, a.n_out, a.commit_cap, hdr, rf);
  count_launches(5);
  return cudaGetLastError();
}

cudaError_t launch_verify(const dspark_verify_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s) {
  if (a.dims.dtype == DSPARK_BF16) return launch_verify_t<__nv_bfloat16>(a, ws, L, s);
  return launch_verify_t<float>(a, ws, L, s);
}

}  // namespace dspark
