// Fitting of the Sequential Temperature Scaling temperatures.
//
// [DSpark] 方法细节, "事后校准（Post-hoc Calibration）": on held-out draft blocks the
// temperatures are chosen left to right, one per position, each by a 1-D grid
// search that minimises the expected calibration error (ECE) of the calibrated
// cumulative product prod_{i<=k} c'_i, the earlier positions held at the
// temperatures already chosen.
//
// ECE is the binned estimate: M equal-width bins on [0, 1] (left-closed, p = 1
// in the last), ECE = (1/N) sum_m |sum_{n in bin m} (y_n - p_n)|, where y_n = 1
// when block n's first k draft tokens were all accepted.
//
// Per position k, two launches:
//   k_sts_hist    every (block, candidate) pair: c' = fp32(sigmoid(z / tau_g))
//                 (fp64 sigmoid), p = fp32(P_{k-1} c'), bin floor(p M); per CTA
//                 private histograms in shared memory (one column per thread, no
//                 atomics), merged into the global table with one atomic per
//                 (bin, candidate).  Before that the CTA extends its blocks'
//                 running products by the temperature position k-1 received.
//   k_sts_select  ECE of every candidate from the table (exact integers), the
//                 first minimum, the chosen temperature.
// The prediction sums are kept in 2^-40 fixed point, so the table adds are exact
// and order-free: the ECE of every candidate is within 2^-41 of the exact value
// for the fp32 predictions, and the choice is deterministic.
//
// c' here comes from a double-float (pairs of fp32) sigmoid on the fp32 pipe,
// with relative error about 2^-47 |t| + 2^-46 against the exact sigmoid (|t| =
// |z| / tau <= 64; beyond, and for non-finite input, the fp64 sigmoid the
// scheduler uses).  Its fp32 rounding is the correctly rounded value except
// where the exact sigmoid lies within that error of an fp32 rounding midpoint:
// a changed c' moves one prediction by one ulp (an ECE change below 1e-7 / N),
// and moves it across a bin edge only if it also sits within an ulp of that
// edge.  Steps (the exponential by Tang's table method, "Table-driven
// implementation of the exponential function in IEEE floating-point
// arithmetic", ACM TOMS 1989):
//   t = z (1/tau)                 1/tau as a double-float, product exact in hi
//   |t| = n ln2/64 + r            n = rint(|t| 64/ln2), ln2/64 split in three
//                                 fp32 parts (the first with 11 bits: n times it
//                                 is exact), |r| <= ln2/128
//   e^-|t| = 2^-(n div 64) 2^-(n mod 64)/64 e^-r, the middle factor from a
//                                 64-entry double-float table, e^-r by its Taylor
//                                 series to degree 5 (the r^2 term in double-float)
//   1/(1 + w) by an approximate fp32 reciprocal y0 and the correction
//                                 y0 (1 + e + e^2), e = 1 - (1 + w) y0.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "dspark.h"
#include "internal.h"
#include "sts_sigmoid.cuh"

namespace dspark {

namespace {

using namespace sts_df;

constexpr int SF_THREADS = 128;
constexpr int SF_SLAB = 256;     // blocks staged in shared memory at a time
constexpr int SF_FX_BITS = 40;   // fixed-point fraction bits of the prediction sums
constexpr int SEL_THREADS = 1024;

struct StsParams {
  int N, G, n_grid, n_bins, k;
  int lanes;  // sample lanes per CTA: threads t < lanes * cols hold (lane, column)
  int cols;   // candidate columns a lane spans: min(n_grid, SF_THREADS)
  int chunk;  // blocks per CTA
  const float* z;
  const int32_t* L;
  const float* grid;
  float* P;                // [G][N] calibrated running products
  unsigned long long* hp;  // [G][n_bins][n_grid] prediction sums (fixed point)
  unsigned int* hy;        // [G][n_bins][n_grid] accepted-prefix counts
  int32_t* gidx;           // [G] chosen candidate
  float* sts_temp;
  int32_t* grid_index;
  double* ece;
  WsHeader* hdr;
};

// bin floor(p * M) (p = 1 -> M - 1) and round(p * 2^40) of an fp32 p in [0, 1];
// anything not below 1.0f (also inf / NaN) counts as 1.  p M is rounded once;
// when that rounding reached the next integer, the exact p M - m (one fma)
// is negative and the bin steps back.  p 2^40 is exact.
__device__ __forceinline__ void bin_and_fixed(float p, float Mf, int M, int& m, unsigned long long& fx) {
  if (!(p < 1.f)) {
    m = M - 1;
    fx = 1ull << SF_FX_BITS;
    return;
  }
  int q = (int)__fmul_rn(p, Mf);
  if (q > 0 && fmaf(p, Mf, -(float)q) < 0.f) --q;
  m = q;
  fx = (unsigned long long)__float2ll_rn(__fmul_rn(p, 0x1p40f));
}

__global__ void __launch_bounds__(SF_THREADS) k_sts_hist(StsParams a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int M = a.n_bins, NG = a.n_grid, lanes = a.lanes, cols = a.cols;
  const float Mf = (float)M;
  const int entries = lanes * M * NG;
  unsigned long long* hist_p = reinterpret_cast<unsigned long long*>(smem);
  unsigned int* hist_y = reinterpret_cast<unsigned int*>(hist_p + entries);
  float* zs = reinterpret_cast<float*>(hist_y + entries);
  float* ps = zs + SF_SLAB;
  unsigned int* ys = reinterpret_cast<unsigned int*>(ps + SF_SLAB);
  __shared__ float2 T64[64];  // 2^(-j/64) as (hi, lo)
  const int t = threadIdx.x;
  for (int e = t; e < entries; e += SF_THREADS) {
    hist_p[e] = 0;
    hist_y[e] = 0;
  }
  if (t < 64) {
    const double v = exp2(-(double)t / 64.0);
    const float hi = (float)v;
    T64[t] = make_float2(hi, (float)(v - (double)hi));
  }

  const int k = a.k, G = a.G, N = a.N;
  // the temperature position k-1 received (written by the previous selection)
  float tau_prev = 1.f, bh_prev = 1.f, bl_prev = 0.f;
  double rtau_prev = 1.0;
  if (k > 0) {
    tau_prev = a.grid[a.gidx[k - 1]];
    rtau_prev = 1.0 / (double)tau_prev;
    bh_prev = (float)rtau_prev;
    bl_prev = (float)(rtau_prev - (double)bh_prev);
  }
  const bool active = t < lanes * cols;
  const int lane = active ? t / cols : 0;
  const int col = active ? t - lane * cols : 0;

  const int begin = blockIdx.x * a.chunk;
  const int end = min(N, begin + a.chunk);
  for (int base = begin; base < end; base += SF_SLAB) {
    const int cnt = min(SF_SLAB, end - base);
    __syncthreads();  // the previous slab is consumed (and the histograms zeroed)
    for (int i = t; i < cnt; i += SF_THREADS) {
      const int n = base + i;
      const size_t row = (size_t)n * G;
      int len = a.L[n];
      if (len < 0 || len > G) {
        if (k == 0) report_error(a.hdr, DSPARK_BAD_INPUT, n);
        len = len < 0 ? 0 : G;
      }
      float pp = 1.f;
      if (k > 0) {
        const float before = k >= 2 ? a.P[(size_t)(k - 2) * N + n] : 1.f;
        pp = __fmul_rn(before, sigmoid_df(a.z[row + k - 1], tau_prev, bh_prev, bl_prev, rtau_prev, T64));
        a.P[(size_t)(k - 1) * N + n] = pp;
      }
      zs[i] = a.z[row + k];
      ps[i] = pp;
      ys[i] = len >= k + 1 ? 1u : 0u;
    }
    __syncthreads();
    if (active) {
      for (int g = col; g < NG; g += cols) {
        const float tau = a.grid[g];
        const double rt = 1.0 / (double)tau;
        const float bh = (float)rt, bl = (float)(rt - (double)bh);
        unsigned long long* hp = hist_p + (size_t)lane * M * NG + g;
        unsigned int* hy = hist_y + (size_t)lane * M * NG + g;
        // two samples per iteration: their sigmoids are independent; the
        // histogram updates then go in sample order (they may hit one bin)
        int i = lane;
#pragma unroll 1
        for (; i + lanes < cnt; i += 2 * lanes) {
          const int i1 = i + lanes;
          const float c0 = sigmoid_df(zs[i], tau, bh, bl, rt, T64);
          const float c1 = sigmoid_df(zs[i1], tau, bh, bl, rt, T64);
          int m0, m1;
          unsigned long long f0, f1;
          bin_and_fixed(__fmul_rn(ps[i], c0), Mf, M, m0, f0);
          bin_and_fixed(__fmul_rn(ps[i1], c1), Mf, M, m1, f1);
          hp[(size_t)m0 * NG] += f0;
          hy[(size_t)m0 * NG] += ys[i];
          hp[(size_t)m1 * NG] += f1;
          hy[(size_t)m1 * NG] += ys[i1];
        }
        if (i < cnt) {
          const float c = sigmoid_df(zs[i], tau, bh, bl, rt, T64);
          int m;
          unsigned long long fx;
          bin_and_fixed(__fmul_rn(ps[i], c), Mf, M, m, fx);
          hp[(size_t)m * NG] += fx;
          hy[(size_t)m * NG] += ys[i];
        }
      }
    }
  }
  __syncthreads();
  unsigned long long* gp = a.hp + (size_t)k * M * NG;
  unsigned int* gy = a.hy + (size_t)k * M * NG;
  for (int e = t; e < M * NG; e += SF_THREADS) {
    unsigned long long sp = 0;
    unsigned int sy = 0;
    for (int l = 0; l < lanes; ++l) {
      sp += hist_p[(size_t)l * M * NG + e];
      sy += hist_y[(size_t)l * M * NG + e];
    }
    if (sp) atomicAdd(gp + e, sp);
    if (sy) atomicAdd(gy + e, sy);
  }
}

__global__ void __launch_bounds__(SEL_THREADS) k_sts_select(StsParams a) {
  __shared__ long long s_num[SEL_THREADS / 32];
  __shared__ int s_idx[SEL_THREADS / 32];
  const int k = a.k, M = a.n_bins, NG = a.n_grid;
  const int t = threadIdx.x;
  const unsigned long long* gp = a.hp + (size_t)k * M * NG;
  const unsigned int* gy = a.hy + (size_t)k * M * NG;
  const double denom = a.N > 0 ? (double)a.N * (double)(1ull << SF_FX_BITS) : 1.0;
  long long best = -1;
  int best_g = 0;
  for (int g = t; g < NG; g += SEL_THREADS) {
    if (k == 0) {
      const float tau = a.grid[g];
      if (!(tau > 0.f) || !(tau < __int_as_float(0x7f800000))) report_error(a.hdr, DSPARK_BAD_INPUT, g);
    }
    long long num = 0;  // sum_m |y_m 2^40 - p_m|, exact: below N 2^40 < 2^63
    for (int m = 0; m < M; ++m) {
      const long long d = ((long long)gy[(size_t)m * NG + g] << SF_FX_BITS) - (long long)gp[(size_t)m * NG + g];
      num += d < 0 ? -d : d;
    }
    a.ece[(size_t)k * NG + g] = (double)num / denom;
    if (best < 0 || num < best) {  // g rises within a thread: keeps the first minimum
      best = num;
      best_g = g;
    }
  }
  // block-wide first minimum of (num, g)
  const int lane = t & 31, w = t >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const long long on = __shfl_down_sync(0xffffffffu, best, off);
    const int og = __shfl_down_sync(0xffffffffu, best_g, off);
    if (on >= 0 && (best < 0 || on < best || (on == best && og < best_g))) {
      best = on;
      best_g = og;
    }
  }
  if (lane == 0) {
    s_num[w] = best;
    s_idx[w] = best_g;
  }
  __syncthreads();
  if (t == 0) {
    for (int i = 1; i < SEL_THREADS / 32; ++i) {
      const long long on = s_num[i];
      const int og = s_idx[i];
      if (on >= 0 && (best < 0 || on < best || (on == best && og < best_g))) {
        best = on;
        best_g = og;
      }
    }
    a.gidx[k] = best_g;
    a.sts_temp[k] = a.grid[best_g];
    if (a.grid_index) a.grid_index[k] = best_g;
  }
}

}  // namespace

StsLayout sts_layout(int N, int G, int n_grid, int n_bins) {
  StsLayout L;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t bytes) {
    off = align_up(off, 256);
    const size_t at = off;
    off += bytes;
    return at;
  };
  const size_t table = (size_t)G * n_bins * n_grid;
  L.hp = take(table * sizeof(unsigned long long));
  L.hy = take(table * sizeof(unsigned int));
  L.table_end = off;
  L.P = take((size_t)G * N * sizeof(float));
  L.gidx = take((size_t)G * sizeof(int32_t));
  L.total = align_up(off, 256);
  return L;
}

static int sts_lanes(int n_grid) { return n_grid >= SF_THREADS ? 1 : SF_THREADS / n_grid; }

size_t sts_hist_smem_bytes(int n_grid, int n_bins) {
  const size_t entries = (size_t)sts_lanes(n_grid) * n_bins * n_grid;
  return entries * (sizeof(unsigned long long) + sizeof(unsigned int)) + SF_SLAB * 3 * sizeof(float);
}

cudaError_t launch_sts_fit(const dspark_sts_fit_args& a, uint8_t* ws, const StsLayout& L, cudaStream_t s) {
  cudaError_t e = ensure_smem_limit((const void*)k_sts_hist,
                                    (int)sts_hist_smem_bytes(SF_THREADS, DSPARK_STS_MAX_TABLE / SF_THREADS));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;  // of the current device
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  StsParams p{};
  p.N = a.N;
  p.G = a.gamma;
  p.n_grid = a.n_grid;
  p.n_bins = a.n_bins;
  p.lanes = sts_lanes(a.n_grid);
  p.cols = a.n_grid < SF_THREADS ? a.n_grid : SF_THREADS;
  p.z = a.conf_logit;
  p.L = a.accept_len;
  p.grid = a.grid;
  p.P = reinterpret_cast<float*>(ws + L.P);
  p.hp = reinterpret_cast<unsigned long long*>(ws + L.hp);
  p.hy = reinterpret_cast<unsigned int*>(ws + L.hy);
  p.gidx = reinterpret_cast<int32_t*>(ws + L.gidx);
  p.sts_temp = a.sts_temp;
  p.grid_index = a.grid_index;
  p.ece = a.ece;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  if ((e = cudaMemsetAsync(ws + L.hp, 0, L.table_end - L.hp, s)) != cudaSuccess) return e;

  const size_t smem = sts_hist_smem_bytes(a.n_grid, a.n_bins);
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_sts_hist, SF_THREADS, smem)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // every CTA resident at once, each with an equal share of the blocks (at
  // least 32 of them, so small sets do not spread over idle CTAs)
  int ctas = sms * per_sm;
  ctas = (int)std::min<long long>(ctas, std::max<long long>(1, ((long long)a.N + 31) / 32));
  p.chunk = (a.N + ctas - 1) / ctas;
  int launches = 0;
  for (int k = 0; k < a.gamma; ++k) {
    p.k = k;
    if (a.N > 0) {
      k_sts_hist<<<ctas, SF_THREADS, smem, s>>>(p);
      ++launches;
    }
    k_sts_select<<<1, SEL_THREADS, 0, s>>>(p);
    ++launches;
  }
  count_launches(launches);
  return cudaGetLastError();
}

}  // namespace dspark
