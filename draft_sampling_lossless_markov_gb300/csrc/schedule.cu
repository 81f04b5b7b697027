// Sequential Temperature Scaling, the hardware-aware prefix scheduler and the
// flattened verify batch, as one CTA of 1024 threads.
//
// [DSpark] 方法细节, "事后校准（Post-hoc Calibration）": c'_k = sigmoid(z_k / tau_k).
// [DSpark] 方法细节, "硬件感知前缀调度器" / "贪心求解与因果性保证", Algorithm 1:
// a_{r,j} = prod_{i<=j} c'_{r,i}; candidates (a > 0) sorted by a descending;
// Theta_i = (B + sum of the first i sorted a) * SPS[B + i]; admit until the first
// Theta_i <= Theta_{i-1}.
// [DSpark] 补充细节, "高吞吐量与低延迟推理": kept prefixes flattened with a
// marker tensor.
//
// Up to 8192 slots (B rounded up to a power of two, times gamma rounded up to
// a power of two) the schedule runs in one CTA's shared memory,
// k_schedule_smem:
//   1. c' for every candidate (a double-float sigmoid on the fp32 pipe, with
//      the fp64 sigmoid deciding the rare values that lie near an fp32
//      rounding boundary, so c' is the fp32 rounding of the fp64 sigmoid), a
//      (the fp32 running product), sort keys key = ~bits(a) for a > 0 (ascending
//      key = descending a), 0xFFFFFFFF else, with the index r * gamma + j;
//      above kFusedKeys candidates k_sched_prep (many CTAs, one thread per
//      candidate) does this step and writes the keys to the workspace;
//   2. one sorted run per request merged pairwise into one;
//   3. fp64 Theta along the sorted path (exact fixed-point survival sums),
//      first non-increase;
//   4. l_r by atomic max over the admitted candidates;
//   5. offsets by a block scan of 1 + l_r; flatten + markers.
// Above 8192 slots k_sched_prep and k_schedule (one CTA of 1024 threads, at
// most 65536 candidates) sort the keys by a stable LSD radix sort (4 passes of
// 8 bits; stability keeps equal a in (r, j) index order) before steps 3-5.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sts_sigmoid.cuh"

namespace dspark {

constexpr int SCH_THREADS = 1024;
constexpr int SCH_WARPS = SCH_THREADS / 32;

// 2^(-j/64), j = 0..63, as double-float (hi, lo) pairs for the double-float
// sigmoid: built once on the host, passed by value to the kernels.
struct DfTable {
  float2 t[64];
};

static const DfTable& df_table() {
  static DfTable tab;
  static std::once_flag once;
  std::call_once(once, [] {
    for (int j = 0; j < 64; ++j) {
      const double v = std::exp2(-(double)j / 64.0);
      const float hi = (float)v;
      tab.t[j] = make_float2(hi, (float)(v - (double)hi));
    }
  });
  return tab;
}

// Per-position STS constants in shared memory: tau, 1/tau as a double-float
// (hi, lo) and in fp64, and the 2^(-j/64) table of the double-float sigmoid.
struct StsConsts {
  float4 tau[DSPARK_MAX_GAMMA];  // (tau, 1/tau hi, 1/tau lo, -)
  double rt[DSPARK_MAX_GAMMA];
  float2 T64[64];
};

// Filled by the first max(64, gamma) threads; the caller syncs before use.
__device__ __forceinline__ void sts_consts_init(StsConsts& c, const float* sts_temp, int G, const DfTable& tab) {
  const int t = threadIdx.x;
  if (t < 64) c.T64[t] = tab.t[t];
  if (t < G) {
    const float tau = sts_temp[t];
    const double rt = 1.0 / (double)tau;
    const float bh = (float)rt;
    c.tau[t] = make_float4(tau, bh, (float)(rt - (double)bh), 0.f);
    c.rt[t] = rt;
  }
}

// calibrated confidence of position j: the fp32 rounding of the fp64 sigmoid of z / tau_j
__device__ __forceinline__ float sts_conf(const StsConsts& c, float z, int j) {
  const float4 tj = c.tau[j];
  return sts_df::sts_sigmoid_exact32(z, tj.x, tj.y, tj.z, c.rt[j], c.T64);
}

// block-wide exclusive scan of one u32 per thread; returns the exclusive prefix
__device__ __forceinline__ uint32_t block_excl_scan_u32(uint32_t v, uint32_t* sm, uint32_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) sm[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t y = sm[lane];
    uint32_t z = y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += t;
    }
    sm[lane] = z - y;  // exclusive prefix of warp totals
    if (lane == 31) sm[32] = z;
  }
  __syncthreads();
  const uint32_t res = sm[wid] + x - v;
  total = sm[32];
  __syncthreads();
  return res;
}

__device__ __forceinline__ double block_excl_scan_f64(double v, double* sm, double& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  double x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) sm[wid] = x;
  __syncthreads();
  if (wid == 0) {
    double z = sm[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += t;
    }
    double ze = __shfl_up_sync(0xffffffffu, z, 1);
    sm[lane] = (lane == 0) ? 0.0 : ze;
    if (lane == 31) sm[32] = z;
  }
  __syncthreads();
  double xe = __shfl_up_sync(0xffffffffu, x, 1);  // exclusive prefix within the warp
  if (lane == 0) xe = 0.0;
  const double res = sm[wid] + xe;
  total = sm[32];
  __syncthreads();
  return res;
}

constexpr int PREP_THREADS = 256;

__device__ __forceinline__ unsigned sched_ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t sched_globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One CTA covers floor(256 / gamma) whole requests: each thread calibrates one
// (request, position) confidence, then one thread per request forms the
// left-to-right fp32 products and writes the sort keys.
// In the asynchronous mode the earlier step's confidences get the same
// treatment into (k1, v1).
__global__ void __launch_bounds__(PREP_THREADS) k_sched_prep(dspark_sched_args a, uint32_t* __restrict__ k0,
                                                             uint32_t* __restrict__ v0, uint32_t* __restrict__ k1,
                                                             uint32_t* __restrict__ v1, const __grid_constant__ DfTable tab) {
  __shared__ float cs[PREP_THREADS];
  __shared__ StsConsts sc;
  const int B = a.B, G = a.gamma;
  sts_consts_init(sc, a.sts_temp, G, tab);
  __syncthreads();
  const int rb = PREP_THREADS / G;
  const int t = threadIdx.x;
  const int lr = t / G, j = t - lr * G;
  const int r = blockIdx.x * rb + lr;
  const bool valid = lr < rb && r < B;
  const int sets = a.mode == DSPARK_SCHED_ASYNC_TOPK ? 2 : 1;
  for (int set = 0; set < sets; ++set) {
    const float* z = set == 0 ? a.conf_logit : a.conf_logit_prev;
    uint32_t* kk = set == 0 ? k0 : k1;
    uint32_t* vv = set == 0 ? v0 : v1;
    if (set) __syncthreads();  // the products of the first set have read cs
    if (valid) cs[t] = sts_conf(sc, z[(size_t)r * G + j], j);
    __syncthreads();
    if (valid && j == 0) {
      float run = 1.f;
      for (int jj = 0; jj < G; ++jj) {
        run = __fmul_rn(run, cs[t + jj]);
        const int idx = r * G + jj;
        kk[idx] = run > 0.f ? ~__float_as_uint(run) : 0xFFFFFFFFu;
        vv[idx] = (uint32_t)idx;
        if (set == 0 && a.surv) a.surv[idx] = run;
      }
      if (set == 0) a.ell[r] = (a.mode == DSPARK_SCHED_OFF) ? G : 0;
    }
  }
}

// fused_keys: this CTA forms the keys itself (k_sched_prep's arithmetic, one
// request per thread at a time) instead of reading k_sched_prep's; dep: as
// for k_schedule_smem (launched behind the draft kernel, beside its last sweep).
__global__ void __launch_bounds__(SCH_THREADS, 1) k_schedule(dspark_sched_args a, uint32_t* __restrict__ k0,
                                                             uint32_t* __restrict__ k1, uint32_t* __restrict__ v0,
                                                             uint32_t* __restrict__ v1, int fused_keys,
                                                             const __grid_constant__ DfTable tab,
                                                             const unsigned* dep, unsigned dep_target,
                                                             WsHeader* hdr) {
  __shared__ uint32_t hist[256 * SCH_WARPS];  // [digit][warp], digit-major
  __shared__ uint32_t sm_u[40];
  __shared__ double sm_d[40];
  __shared__ int s_first;
  __shared__ double s_theta_best;
  __shared__ StsConsts sc;

  const int B = a.B, G = a.gamma, n = B * G;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (dep) {
    if (tid == 0) {
      const uint64_t t0 = sched_globaltimer_ns();
      int ok = 1;
      while (sched_ld_acquire(dep) < dep_target) {
        if (sched_globaltimer_ns() - t0 > 2000000000ull) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
      if (!ok) report_error(hdr, DSPARK_TIMEOUT, -1);
      s_first = ok;
    }
    __syncthreads();
    if (!s_first) return;
  }
  if (fused_keys) {
    sts_consts_init(sc, a.sts_temp, G, tab);
    __syncthreads();
    for (int r = tid; r < B; r += SCH_THREADS) {
      float run = 1.f;
      for (int jj = 0; jj < G; ++jj) {
        const int idx = r * G + jj;
        run = __fmul_rn(run, sts_conf(sc, a.conf_logit[idx], jj));
        k0[idx] = run > 0.f ? ~__float_as_uint(run) : 0xFFFFFFFFu;
        v0[idx] = (uint32_t)idx;
        if (a.surv) a.surv[idx] = run;
      }
      a.ell[r] = (a.mode == DSPARK_SCHED_OFF) ? G : 0;
    }
    __syncthreads();  // the keys and l_r = 0, for every thread of the CTA
  }

  // ---- candidates: keys written by k_sched_prep; a > 0 unless the key is all ones ----
  uint32_t ncand_local = 0;
  for (int i = tid; i < n; i += SCH_THREADS) ncand_local += (k0[i] != 0xFFFFFFFFu);
  uint32_t ncand;
  block_excl_scan_u32(ncand_local, sm_u, ncand);

  if (a.mode != DSPARK_SCHED_OFF) {
    // ---- 2. stable LSD radix sort, 4 passes of 8 bits ----
    const int seg = ((n + SCH_WARPS - 1) / SCH_WARPS + 31) & ~31;
    const int w_lo = min(wid * seg, n), w_hi = min(w_lo + seg, n);
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 8 * pass;
      const uint32_t* sk = (pass & 1) ? k1 : k0;
      const uint32_t* sv = (pass & 1) ? v1 : v0;
      uint32_t* dk = (pass & 1) ? k0 : k1;
      uint32_t* dv = (pass & 1) ? v0 : v1;
      for (int i = tid; i < 256 * SCH_WARPS; i += SCH_THREADS) hist[i] = 0;
      __syncthreads();
      for (int base = w_lo; base < w_hi; base += 32) {
        const int idx = base + lane;
        const bool valid = idx < w_hi;
        const uint32_t d = valid ? ((sk[idx] >> shift) & 255u) : 256u;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        if (valid && lane == __ffs(peers) - 1) hist[d * SCH_WARPS + wid] += __popc(peers);
        __syncwarp();
      }
      __syncthreads();
      // exclusive scan over (digit, warp) in digit-major order: 8 entries per thread
      {
        uint32_t loc[8], s = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          loc[e] = hist[tid * 8 + e];
          s += loc[e];
        }
        uint32_t tot;
        uint32_t p = block_excl_scan_u32(s, sm_u, tot);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          hist[tid * 8 + e] = p;
          p += loc[e];
        }
      }
      __syncthreads();
      for (int base = w_lo; base < w_hi; base += 32) {
        const int idx = base + lane;
        const bool valid = idx < w_hi;
        const uint32_t key = valid ? sk[idx] : 0u;
        const uint32_t val = valid ? sv[idx] : 0u;
        const uint32_t d = valid ? ((key >> shift) & 255u) : 256u;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        if (valid) {
          const uint32_t dst = hist[d * SCH_WARPS + wid] + __popc(peers & lt_mask);
          dk[dst] = key;
          dv[dst] = val;
        }
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) hist[d * SCH_WARPS + wid] += __popc(peers);
        __syncwarp();
      }
      __syncthreads();
    }
    // sorted keys / values are back in k0 / v0 (even number of passes)

    // ---- 3. Theta along the sorted path, first non-increase ----
    const int nc = (int)ncand;
    const int ch = (nc + SCH_THREADS - 1) / SCH_THREADS;
    const int c_lo = min(tid * ch, nc), c_hi = min(c_lo + ch, nc);
    double loc = 0.0;
    for (int i = c_lo; i < c_hi; ++i) loc += (double)__uint_as_float(~k0[i]);
    double tot;
    const double pre = block_excl_scan_f64(loc, sm_d, tot);
    if (tid == 0) s_first = nc + 1;
    __syncthreads();
    {
      double S = pre;
      double theta_prev = ((double)B + S) * a.sps[B + c_lo];
      for (int i = c_lo; i < c_hi; ++i) {  // sorted position i is candidate number i + 1
        S += (double)__uint_as_float(~k0[i]);
        const double theta = ((double)B + S) * a.sps[B + i + 1];
        if (!(theta > theta_prev)) {
          atomicMin(&s_first, i + 1);
          break;
        }
        theta_prev = theta;
      }
    }
    __syncthreads();
    const int nstar = s_first - 1;  // admitted candidates
    // Theta of the kept set: recomputed by the thread that owns candidate nstar
    if (nstar == 0) {
      if (tid == 0) s_theta_best = (double)B * a.sps[B];
    } else if (nstar - 1 >= c_lo && nstar - 1 < c_hi) {
      double S = pre;
      for (int i = c_lo; i < nstar; ++i) S += (double)__uint_as_float(~k0[i]);
      s_theta_best = ((double)B + S) * a.sps[B + nstar];
    }
    // ---- 4. l_r = number of admitted (r, .) candidates (= largest admitted j) ----
    for (int i = tid; i < nstar; i += SCH_THREADS) {
      const uint32_t v = v0[i];
      atomicMax(&a.ell[v / G], (int)(v % G) + 1);
    }
    __syncthreads();
    if (tid == 0) *a.theta_best = s_theta_best;
  } else {
    if (tid == 0) *a.theta_best = 0.0;
  }
  __syncthreads();

  // ---- 5. offsets and the flattened batch ----
  const int chb = (B + SCH_THREADS - 1) / SCH_THREADS;
  const int b_lo = min(tid * chb, B), b_hi = min(b_lo + chb, B);
  uint32_t cnt = 0;
  for (int r = b_lo; r < b_hi; ++r) cnt += 1u + (uint32_t)a.ell[r];
  uint32_t nv;
  uint32_t off = block_excl_scan_u32(cnt, sm_u, nv);
  for (int r = b_lo; r < b_hi; ++r) {
    a.offsets[r] = (int)off;
    const int L = a.ell[r];
    a.flat_tok[off] = a.anchor[r];
    a.mark_req[off] = r;
    a.mark_pos[off] = 0;
    for (int j = 1; j <= L; ++j) {
      a.flat_tok[off + j] = a.tokens[(size_t)r * G + j - 1];
      a.mark_req[off + j] = r;
      a.mark_pos[off + j] = j;
    }
    off += 1u + (uint32_t)L;
  }
  const int cap = B * (1 + G);
  for (int i = (int)nv + tid; i < cap; i += SCH_THREADS) {
    a.flat_tok[i] = -1;
    a.mark_req[i] = -1;
    a.mark_pos[i] = -1;
  }
  if (tid == 0) {
    a.offsets[B] = (int)nv;
    *a.n_verify = (int)nv;
  }
}

// Up to kSmemSortMax slots the whole schedule runs out of shared memory.  A
// request's candidates are already in sort order (its survival products only
// shrink along the prefix, so their keys only grow, and its indices grow), so
// the (key, index) pairs are laid out as one sorted run per request, padded to
// R = 2^ceil(log2 gamma) slots, and merged pairwise (merge path: an element's
// place is its rank in its own run plus its rank in the partner run) until one
// run remains; the 64-bit (key, index) order is the radix sort's stable order
// (ties in a stay in (r, j) index order).  Then the same Theta scan, l_r and
// flatten as k_schedule.
constexpr int kSmemSortMax = 8192;
constexpr int kFusedKeys = 2048;  // candidates up to which k_schedule_smem calibrates them itself
static_assert(kSmemSortMax <= 8 * 1024, "merge_runs keeps eight elements per thread");
constexpr int kPrefetchTok = 8;  // draft lengths whose tokens k_schedule_smem loads at its start
constexpr size_t kSmemSchedMax = 200 * 1024;  // dynamic shared memory of k_schedule_smem

__device__ __forceinline__ float key_to_a(uint64_t kv) { return __uint_as_float(~(uint32_t)(kv >> 32)); }

// a (in (0, 1], from the sort key) as a fixed-point integer with 50 fraction
// bits, by integer operations on its fp32 fields: exact for a >= 2^-27,
// truncated below (by less than 2^-50 per candidate), 0 for subnormals.  Sums
// of these are exact in 64 unsigned bits for up to 2^14 candidates (a <= 1), so
// the running survival sum of the Theta scan needs no fp64 adds; the
// truncation moves B + sum by less than gamma 2^-50 relative.
__device__ __forceinline__ unsigned long long key_to_fix(uint64_t kv) {
  const uint32_t bits = ~(uint32_t)(kv >> 32);
  const int e = (int)((bits >> 23) & 0xFFu);
  if (e == 0) return 0;
  const unsigned long long m = (unsigned long long)((bits & 0x7FFFFFu) | 0x800000u);
  const int sh = e - 100;  // m 2^(e - 150) 2^50
  return sh >= 0 ? (m << sh) : (sh > -64 ? (m >> -sh) : 0);
}
constexpr double kFixUnit = 8.8817841970012523233890533447265625e-16;  // 2^-50
static_assert(kSmemSortMax <= (1 << 14), "fixed-point survival sums hold 2^14 candidates");

__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v, unsigned long long* sm,
                                                                  unsigned long long& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) sm[wid] = x;
  __syncthreads();
  if (wid == 0) {
    unsigned long long z = sm[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += t;
    }
    const unsigned long long ze = __shfl_up_sync(0xffffffffu, z, 1);
    sm[lane] = (lane == 0) ? 0 : ze;
    if (lane == 31) sm[32] = z;
  }
  __syncthreads();
  unsigned long long xe = __shfl_up_sync(0xffffffffu, x, 1);  // exclusive prefix within the warp
  if (lane == 0) xe = 0;
  const unsigned long long res = sm[wid] + xe;
  total = sm[32];
  __syncthreads();
  return res;
}

// Theta_j = (B + S_j 2^-50) SPS[B + j] in fp64, the value the sorted-path scan
// compares
__device__ __forceinline__ double theta64(int B, unsigned long long S, double sps) {
  return ((double)B + (double)S * kFixUnit) * sps;
}

// The same in fp32, with a relative error below 2^-21 for a positive SPS
// entry in fp32's normal range, else 0: S rounded to fp32 (one rounding), the
// sum with B (one), the SPS entry truncated to fp32 by its bit fields (below
// 2^-23), the product (one).  No fp64 arithmetic.
__device__ __forceinline__ float theta32(int B, unsigned long long S, double sps) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(sps);
  const int e = (int)((b >> 52) & 0x7FF) - 1023 + 127;
  if ((b >> 63) || e <= 0 || e >= 255) return 0.f;
  const float s32 = __uint_as_float(((unsigned)e << 23) | (unsigned)((b >> 29) & 0x7FFFFFu));
  return __fmul_rn(__fadd_rn((float)B, __fmul_rn(__ull2float_rn(S), 0x1p-50f)), s32);
}

// Theta_{j+1} > Theta_j as the fp64 values compare: decided in fp32 when the
// two fp32 values differ by more than 2^-19 relative (twice the bound on their
// combined error), by the fp64 values otherwise
__device__ __forceinline__ bool theta_rises(int B, unsigned long long S0, double sps0, float t0,
                                            unsigned long long S1, double sps1, float t1) {
  constexpr float kLo = 1e-30f, kHi = 1e30f;
  if (t0 > kLo && t0 < kHi && t1 > kLo && t1 < kHi) {
    if (t1 > __fmul_rn(t0, 1.f + 0x1p-19f)) return true;
    if (t1 < __fmul_rn(t0, 1.f - 0x1p-19f)) return false;
  }
  return theta64(B, S1, sps1) > theta64(B, S0, sps0);
}

// Merges sorted runs of length run0 (a power of two) in a[0, n_pad) (n_pad /
// run0 a power of two, all values distinct, n_pad <= kSmemSortMax) into one
// sorted run; b is scratch of the same size.  Each pass merges pairs of runs
// of width w into runs of 2w along the merge path: thread t writes outputs
// t EPT .. t EPT + EPT - 1, finding by one halving search how many of the
// outputs before its first come from the left run (its diagonal's split),
// then taking the smaller head of the two runs EPT times.  Returns the buffer
// that holds the result.
template <int EPT>  // outputs per thread: n_pad <= EPT * SCH_THREADS
__device__ uint64_t* merge_runs_t(uint64_t* a, uint64_t* b, int n_pad, int run0) {
  const int o0 = threadIdx.x * EPT;
  const bool act = o0 < n_pad;
  for (int w = run0; w < n_pad; w <<= 1) {
    if (act) {
      int blk = o0 & ~(2 * w - 1);  // the pair of runs: [blk, blk + w) and [blk + w, blk + 2w)
      const int d = o0 - blk;
      const uint64_t* L = a + blk;
      const uint64_t* Rr = L + w;
      int lo = max(0, d - w), hi = min(d, w);
      while (lo < hi) {  // the split: L[0, ia) and Rr[0, d - ia) precede output d
        const int mid = (lo + hi) >> 1;
        if (L[mid] < Rr[d - 1 - mid])
          lo = mid + 1;
        else
          hi = mid;
      }
      int ia = lo, ib = d - lo;
      uint64_t va = ia < w ? L[ia] : ~0ull, vb = ib < w ? Rr[ib] : ~0ull;  // an empty run's head sorts last
#pragma unroll
      for (int k = 0; k < EPT; ++k) {
        if (k > 0 && ((o0 + k) & (2 * w - 1)) == 0) {
          // (2w < EPT) the next pair of runs starts inside this thread's outputs
          blk += 2 * w;
          L = a + blk;
          Rr = L + w;
          ia = 0;
          ib = 0;
          va = L[0];
          vb = Rr[0];
        }
        const bool from_l = va < vb;
        b[o0 + k] = from_l ? va : vb;
        if (from_l) {
          ++ia;
          va = ia < w ? L[ia] : ~0ull;
        } else {
          ++ib;
          vb = ib < w ? Rr[ib] : ~0ull;
        }
      }
    }
    __syncthreads();
    uint64_t* t = a;
    a = b;
    b = t;
  }
  return a;
}

__device__ uint64_t* merge_runs(uint64_t* a, uint64_t* b, int n_pad, int run0) {
  if (n_pad <= SCH_THREADS) return merge_runs_t<1>(a, b, n_pad, run0);
  if (n_pad <= 2 * SCH_THREADS) return merge_runs_t<2>(a, b, n_pad, run0);
  if (n_pad <= 4 * SCH_THREADS) return merge_runs_t<4>(a, b, n_pad, run0);
  return merge_runs_t<8>(a, b, n_pad, run0);
}

// slots of the shared-memory schedule: one run of R slots per request, the
// number of runs a power of two
__host__ __device__ inline int sched_run_len(int G) {
  int R = 1;
  while (R < G) R <<= 1;
  return R;
}
__host__ __device__ inline int sched_slots(int B, int G) {
  int nb = 1;
  while (nb < B) nb <<= 1;
  return nb * sched_run_len(G);
}

// Largest value, first index on ties, over the CTA (every thread gets it).
__device__ __forceinline__ void block_argmax_f64(double& v, int& i, double* smv, int* smi) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    if (v2 > v || (v2 == v && i2 < i)) {
      v = v2;
      i = i2;
    }
  }
  if (lane == 0) {
    smv[wid] = v;
    smi[wid] = i;
  }
  __syncthreads();
  v = smv[0];
  i = smi[0];
  for (int w = 1; w < SCH_THREADS / 32; ++w)
    if (smv[w] > v || (smv[w] == v && smi[w] < i)) {
      v = smv[w];
      i = smi[w];
    }
  __syncthreads();
}

// dep (may be null): launched behind the draft kernel with programmatic
// stream serialization, so that it runs beside the draft's last sweep; the
// draft's CTAs add 1 to *dep (release) once the confidences and tokens are
// written and let this grid launch only after that, so the wait below finds
// *dep == dep_target at once (it gives up after a bound all the same and
// reports DSPARK_TIMEOUT to hdr).
__global__ void __launch_bounds__(SCH_THREADS, 1) k_schedule_smem(dspark_sched_args a, int n_pad,
                                                                  const __grid_constant__ DfTable tab,
                                                                  const uint32_t* __restrict__ k0,
                                                                  const uint32_t* __restrict__ v0,
                                                                  const uint32_t* __restrict__ k1,
                                                                  const uint32_t* __restrict__ v1, int fused,
                                                                  const unsigned* dep, unsigned dep_target,
                                                                  WsHeader* hdr) {
  // [n_pad] slots, [n_pad] scratch (first holding the calibrated confidences),
  // [B (1 + gamma) + 1] SPS table, [B] l_r
  extern __shared__ uint64_t kv[];
  uint64_t* kv2 = kv + n_pad;
  const int B = a.B, G = a.gamma;
  double* s_sps = reinterpret_cast<double*>(kv2 + n_pad);
  int* s_ell = reinterpret_cast<int*>(s_sps + B * (1 + G) + 1);
  float* s_c = reinterpret_cast<float*>(kv2);  // [B gamma] c', until the merge reuses kv2
  __shared__ uint32_t sm_u[40];
  __shared__ unsigned long long sm_l[40];
  __shared__ double sm_v[32];
  __shared__ int sm_i[32];
  __shared__ int s_first;
  __shared__ double s_theta_best;
  __shared__ StsConsts sc;

  const int tid = threadIdx.x;
  if (dep) {
    if (tid == 0) {
      const uint64_t t0 = sched_globaltimer_ns();
      int ok = 1;
      while (sched_ld_acquire(dep) < dep_target) {
        if (sched_globaltimer_ns() - t0 > 2000000000ull) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
      if (!ok) report_error(hdr, DSPARK_TIMEOUT, -1);
      s_first = ok;
    }
    __syncthreads();
    if (!s_first) return;
  }
  const int R = sched_run_len(G);
  sts_consts_init(sc, a.sts_temp, G, tab);
  // the flatten's inputs for this thread's request, loaded now so that their
  // latency overlaps the sort (the later stores could alias them, so the
  // compiler would not hoist the loads itself)
  const int chb = (B + SCH_THREADS - 1) / SCH_THREADS;
  const int b_lo = min(tid * chb, B), b_hi = min(b_lo + chb, B);
  const bool pre = chb == 1 && G <= kPrefetchTok && b_lo < b_hi;
  int pre_anchor = 0, pre_tok[kPrefetchTok];
  if (pre) {
    pre_anchor = a.anchor[b_lo];
#pragma unroll
    for (int j = 0; j < kPrefetchTok; ++j) pre_tok[j] = j < G ? a.tokens[(size_t)b_lo * G + j] : 0;
  }
  for (int r = tid; r < B; r += SCH_THREADS) s_ell[r] = (a.mode == DSPARK_SCHED_OFF) ? G : 0;
  if (a.mode != DSPARK_SCHED_OFF)
    for (int i = tid; i <= B * (1 + G); i += SCH_THREADS) s_sps[i] = a.sps[i];
  __syncthreads();  // the STS constants
  // c' of every candidate, then one sorted run per request in kv (a request's
  // keys only grow along its prefix, so each run is sorted), padded; returns
  // the number of candidates (a > 0)
  auto build_runs = [&](const float* z, bool write_surv, const uint32_t* kk, const uint32_t* vv) {
    const int n = B * G;
    if (!fused) {
      // keys from k_sched_prep (more candidates than one SM calibrates quickly)
      uint32_t ncand_local = 0;
      for (int i = tid; i < n_pad; i += SCH_THREADS) {
        const int r = i / R, j = i - r * R;
        uint64_t e = (0xFFFFFFFFull << 32) | (0x80000000u + (uint32_t)i);
        if (r < B && j < G) {
          const uint32_t key = kk[r * G + j];
          ncand_local += key != 0xFFFFFFFFu;
          e = ((uint64_t)key << 32) | vv[r * G + j];
        }
        kv[i] = e;
      }
      uint32_t nc;
      block_excl_scan_u32(ncand_local, sm_u, nc);
      return nc;
    }
    for (int i = tid; i < n; i += SCH_THREADS) s_c[i] = sts_conf(sc, z[i], i % G);
    __syncthreads();
    uint32_t ncand_local = 0;
    for (int i = tid; i < n_pad; i += SCH_THREADS) {
      const int r = i / R, j = i - r * R;
      // padding sorts after every candidate and non-candidate, each slot distinct
      uint64_t e = (0xFFFFFFFFull << 32) | (0x80000000u + (uint32_t)i);
      if (r < B && j < G) {
        // a_{r,j}: the left-to-right fp32 product, the same chain for every j
        float run = 1.f;
        for (int jj = 0; jj <= j; ++jj) run = __fmul_rn(run, s_c[r * G + jj]);
        const uint32_t key = run > 0.f ? ~__float_as_uint(run) : 0xFFFFFFFFu;
        ncand_local += key != 0xFFFFFFFFu;
        e = ((uint64_t)key << 32) | (uint32_t)(r * G + j);
        if (write_surv && a.surv) a.surv[r * G + j] = run;
      }
      kv[i] = e;
    }
    uint32_t nc;
    block_excl_scan_u32(ncand_local, sm_u, nc);  // ends with __syncthreads: kv2 (c') is free again
    return nc;
  };
  if (a.mode == DSPARK_SCHED_ASYNC_TOPK) {
    // ---- capacity: the best prefix of the earlier step's sorted path (global search) ----
    const int nprev = (int)build_runs(a.conf_logit_prev, false, k1, v1);
    const uint64_t* prv = merge_runs(kv, kv2, n_pad, R);
    const int chp = (nprev + SCH_THREADS - 1) / SCH_THREADS;
    const int p_lo = min(tid * chp, nprev), p_hi = min(p_lo + chp, nprev);
    unsigned long long loc = 0;
    for (int i = p_lo; i < p_hi; ++i) loc += key_to_fix(prv[i]);
    unsigned long long tot;
    unsigned long long S = block_excl_scan_u64(loc, sm_l, tot);
    double bv = tid == 0 ? (double)B * s_sps[B] : -INFINITY;  // Theta_0: nothing admitted
    int bi = tid == 0 ? 0 : INT_MAX;
    for (int i = p_lo; i < p_hi; ++i) {
      S += key_to_fix(prv[i]);
      const double theta = theta64(B, S, s_sps[B + i + 1]);
      if (theta > bv) {
        bv = theta;
        bi = i + 1;
      }
    }
    block_argmax_f64(bv, bi, sm_v, sm_i);
    const int K = bi;
    // ---- this step: its candidates in order, the first min(K, n) admitted ----
    const int ncur = (int)build_runs(a.conf_logit, true, k0, v0);  // every read of the earlier path ended before the scan's barriers
    const uint64_t* cur = merge_runs(kv, kv2, n_pad, R);
    const int nadm = min(K, ncur);
    unsigned long long sl = 0;
    for (int i = tid; i < nadm; i += SCH_THREADS) {
      const uint32_t v = (uint32_t)cur[i];
      atomicMax(&s_ell[v / G], (int)(v % G) + 1);
      sl += key_to_fix(cur[i]);
    }
    unsigned long long sadm;
    block_excl_scan_u64(sl, sm_l, sadm);
    if (tid == 0) *a.theta_best = theta64(B, sadm, s_sps[B + nadm]);
  } else if (a.mode != DSPARK_SCHED_OFF) {
    const uint32_t ncand = build_runs(a.conf_logit, true, k0, v0);
    // ---- 2. one sorted run: ascending (key, index) = descending a, ties by index ----
    const uint64_t* srt = merge_runs(kv, kv2, n_pad, R);
    // ---- 3. Theta along the sorted path, first non-increase ----
    const int nc = (int)ncand;
    const int ch = (nc + SCH_THREADS - 1) / SCH_THREADS;
    const int c_lo = min(tid * ch, nc), c_hi = min(c_lo + ch, nc);
    // survival sums in fixed point (exact adds); Theta compared as in fp64
    unsigned long long loc = 0;
    for (int i = c_lo; i < c_hi; ++i) loc += key_to_fix(srt[i]);
    unsigned long long tot;
    const unsigned long long pre_s = block_excl_scan_u64(loc, sm_l, tot);
    if (tid == 0) s_first = nc + 1;
    __syncthreads();
    if (c_lo < c_hi) {
      unsigned long long S = pre_s;
      double sp = s_sps[B + c_lo];
      float t_prev = theta32(B, S, sp);
      for (int i = c_lo; i < c_hi; ++i) {  // sorted position i is candidate number i + 1
        const unsigned long long S1 = S + key_to_fix(srt[i]);
        const double sp1 = s_sps[B + i + 1];
        const float t = theta32(B, S1, sp1);
        if (!theta_rises(B, S, sp, t_prev, S1, sp1, t)) {
          atomicMin(&s_first, i + 1);
          break;
        }
        S = S1;
        sp = sp1;
        t_prev = t;
      }
    }
    __syncthreads();
    const int nstar = s_first - 1;  // admitted candidates
    if (nstar == 0) {
      if (tid == 0) s_theta_best = (double)B * s_sps[B];
    } else if (nstar - 1 >= c_lo && nstar - 1 < c_hi) {
      unsigned long long S = pre_s;
      for (int i = c_lo; i < nstar; ++i) S += key_to_fix(srt[i]);
      s_theta_best = theta64(B, S, s_sps[B + nstar]);
    }
    // ---- 4. l_r = number of admitted (r, .) candidates (= largest admitted j) ----
    for (int i = tid; i < nstar; i += SCH_THREADS) {
      const uint32_t v = (uint32_t)srt[i];
      atomicMax(&s_ell[v / G], (int)(v % G) + 1);
    }
    __syncthreads();
    if (tid == 0) *a.theta_best = s_theta_best;
  } else {
    if (a.surv && fused) build_runs(a.conf_logit, true, k0, v0);  // the survival products only
    if (tid == 0) *a.theta_best = 0.0;
  }
  __syncthreads();

  // ---- 5. offsets and the flattened batch ----
  uint32_t cnt = 0;
  for (int r = b_lo; r < b_hi; ++r) cnt += 1u + (uint32_t)s_ell[r];
  uint32_t nv;
  uint32_t off = block_excl_scan_u32(cnt, sm_u, nv);
  if (pre) {
    const int r = b_lo, L = s_ell[r];
    a.ell[r] = L;
    a.offsets[r] = (int)off;
    a.flat_tok[off] = pre_anchor;
    a.mark_req[off] = r;
    a.mark_pos[off] = 0;
#pragma unroll
    for (int j = 1; j <= kPrefetchTok; ++j) {
      if (j <= L) {
        a.flat_tok[off + j] = pre_tok[j - 1];
        a.mark_req[off + j] = r;
        a.mark_pos[off + j] = j;
      }
    }
  } else {
    for (int r = b_lo; r < b_hi; ++r) {
      const int L = s_ell[r];
      a.ell[r] = L;
      a.offsets[r] = (int)off;
      a.flat_tok[off] = a.anchor[r];
      a.mark_req[off] = r;
      a.mark_pos[off] = 0;
      for (int j = 1; j <= L; ++j) {
        a.flat_tok[off + j] = a.tokens[(size_t)r * G + j - 1];
        a.mark_req[off + j] = r;
        a.mark_pos[off + j] = j;
      }
      off += 1u + (uint32_t)L;
    }
  }
  const int cap = B * (1 + G);
  for (int i = (int)nv + tid; i < cap; i += SCH_THREADS) {
    a.flat_tok[i] = -1;
    a.mark_req[i] = -1;
    a.mark_pos[i] = -1;
  }
  if (tid == 0) {
    a.offsets[B] = (int)nv;
    *a.n_verify = (int)nv;
  }
}

static size_t schedule_smem_bytes(int B, int G) {
  // slots, merge scratch, the SPS table and l_r
  return 2 * (size_t)sched_slots(B, G) * sizeof(uint64_t) + ((size_t)B * (1 + G) + 1) * sizeof(double) +
         (size_t)B * sizeof(int);
}

bool schedule_async_supported(int B, int G) {
  return sched_slots(B, G) <= kSmemSortMax && schedule_smem_bytes(B, G) <= kSmemSchedMax;
}

bool schedule_behind_draft_supported(int B, int G) { return (int64_t)B * G <= DSPARK_MAX_SCHED_KEYS; }

cudaError_t launch_schedule_behind_draft(const dspark_sched_args& a, uint8_t* ws, const WsLayout& L,
                                         const unsigned* dep, unsigned dep_target, cudaStream_t s) {
  if (!schedule_behind_draft_supported(a.B, a.gamma)) return cudaErrorNotSupported;
  uint32_t* k0 = reinterpret_cast<uint32_t*>(ws + L.sk0);
  uint32_t* k1 = reinterpret_cast<uint32_t*>(ws + L.sk1);
  uint32_t* v0 = reinterpret_cast<uint32_t*>(ws + L.sv0);
  uint32_t* v1 = reinterpret_cast<uint32_t*>(ws + L.sv1);
  const int n_pad = sched_slots(a.B, a.gamma);
  const bool smem_path = schedule_async_supported(a.B, a.gamma);
  if (smem_path) {
    if (const cudaError_t ae = ensure_smem_limit((const void*)k_schedule_smem, (int)kSmemSchedMax);
        ae != cudaSuccess)
      return ae;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(SCH_THREADS);
  cfg.dynamicSmemBytes = smem_path ? schedule_smem_bytes(a.B, a.gamma) : 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  // the keys calibrated in this one CTA at every size (no k_sched_prep on many
  // SMs): beside the draft's last sweep only one SM is free
  cudaError_t e = smem_path
                      ? cudaLaunchKernelEx(&cfg, k_schedule_smem, a, n_pad, df_table(), (const uint32_t*)k0,
                                           (const uint32_t*)v0, (const uint32_t*)k1, (const uint32_t*)v1, 1, dep,
                                           dep_target, reinterpret_cast<WsHeader*>(ws))
                      : cudaLaunchKernelEx(&cfg, k_schedule, a, k0, k1, v0, v1, 1, df_table(), dep, dep_target,
                                           reinterpret_cast<WsHeader*>(ws));
  if (e != cudaSuccess) return e;
  if (a.n_verify_host) e = cudaMemcpyAsync(a.n_verify_host, a.n_verify, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  return e;
}

cudaError_t launch_schedule(const dspark_sched_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s) {
  uint32_t* k0 = reinterpret_cast<uint32_t*>(ws + L.sk0);
  uint32_t* k1 = reinterpret_cast<uint32_t*>(ws + L.sk1);
  uint32_t* v0 = reinterpret_cast<uint32_t*>(ws + L.sv0);
  uint32_t* v1 = reinterpret_cast<uint32_t*>(ws + L.sv1);
  // every refusal comes before the first launch
  if (a.mode == DSPARK_SCHED_ASYNC_TOPK && !schedule_async_supported(a.B, a.gamma)) return cudaErrorNotSupported;
  const int n_pad = sched_slots(a.B, a.gamma);
  const size_t smem = schedule_smem_bytes(a.B, a.gamma);
  if (n_pad <= kSmemSortMax && smem <= kSmemSchedMax) {
    // up to kFusedKeys candidates one launch does everything (confidences, keys,
    // sort, Theta, flatten); above, k_sched_prep calibrates on many SMs first
    if (const cudaError_t ae = ensure_smem_limit((const void*)k_schedule_smem, (int)kSmemSchedMax); ae != cudaSuccess)
      return ae;
    const int fused = (int64_t)a.B * a.gamma <= kFusedKeys ? 1 : 0;
    if (!fused) {
      const int rb = PREP_THREADS / a.gamma;
      k_sched_prep<<<(a.B + rb - 1) / rb, PREP_THREADS, 0, s>>>(a, k0, v0, k1, v1, df_table());
    }
    k_schedule_smem<<<1, SCH_THREADS, smem, s>>>(a, n_pad, df_table(), k0, v0, k1, v1, fused, nullptr, 0u,
                                                 reinterpret_cast<WsHeader*>(ws));
    count_launches(fused ? 1 : 2);
  } else {
    const int rb = PREP_THREADS / a.gamma;
    k_sched_prep<<<(a.B + rb - 1) / rb, PREP_THREADS, 0, s>>>(a, k0, v0, k1, v1, df_table());
    k_schedule<<<1, SCH_THREADS, 0, s>>>(a, k0, k1, v0, v1, 0, df_table(), nullptr, 0u,
                                         reinterpret_cast<WsHeader*>(ws));
    count_launches(2);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.n_verify_host) e = cudaMemcpyAsync(a.n_verify_host, a.n_verify, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  return e;
}

}  // namespace dspark
