// Tensor-core (tcgen05) draft sampler of the Markov head, sm_103a.
//
// The Markov-head bias of position k is a dense contraction
//     bias[b, v] = E[b, :] . W2[:, v],   E[b] = W1[x_{k-1}]      (B x r x V)
// ([DSpark] 方法细节, "马尔可夫头（Markov head）的实现").  With r = 256 it is
// 2 r = 512 flop per (b, v) against 6 bytes of U read + p_d write, i.e. far
// above the CUDA-core ridge, so it runs on the 5th-generation tensor cores.
//
// One persistent kernel runs all gamma positions of a draft call.  Each
// position takes two passes over the vocabulary, because the exact p_d row
// needs its normaliser before any element can be written and the logits of a
// position do not fit on chip:
//   pass 1  logits -> per-(row, 64-column chunk) partial (max, sum 2^(y-m),
//           argmax) and per-(row, CTA segment) partial; confidence c_k
//   select  one warp per row: row max and sum from the segment partials, the
//           Philox draw, the segment and then the chunk where the CDF crosses
//           u S; greedy rows take the argmax and are done
//   pass 2  recompute the logits, write p_d = 2^(y - m) / S; the CTA that owns
//           the crossing chunk walks it with exactly the values it writes and
//           emits the token and p_d(x_k)
// with grid-wide barriers after pass 1, after the select and after pass 2.
// The TMA producer does not take part in the barriers: U and W2 are inputs, so
// it keeps streaming the next phase's tiles into the rings while the other
// roles wait, and HBM stays busy across the phase boundaries.
//
// Tile: 128 requests (TMEM lanes) x 192 vocabulary columns, K = r.  One
// tcgen05.mma instruction costs about the same for N = 64 and N = 128 and
// reaches the tensor-core peak only near N = 256, so the tile is as wide as
// TMEM allows: E (the A operand, r/2 columns) plus two 192-column fp32
// accumulators fill the 512 columns.
//
//   warp 0    TMA producer, two rings: W2 in K-chunks [64 x 192] and U in
//             tiles [128 x 192] (three 64-column boxes), all 128B-swizzled
//   warp 1    allocates TMEM, issues tcgen05.mma (A = E from TMEM, B = W2
//             K-chunk from shared memory, MN-major, N = 192) into one of the
//             two accumulators, commits to mbarriers
//   warps 2-13 epilogue, three groups of four warps (one per TMEM lane
//             quarter); group g owns the g-th 64-column chunk of every tile.
//             Per position they copy the E rows into TMEM; per tile: TMEM ->
//             registers, + U, then the chunk partial (pass 1) or the p_d row
//             through a per-warp swizzled staging buffer and TMA stores
//             (pass 2).  They also run the select and the grid barriers.
//
// A CTA owns one 128-row M-tile and a contiguous segment of its vocabulary
// tiles; pass 1 walks the segment upward and pass 2 downward, so pass 2 starts
// on the tiles whose lines are the likeliest to still be in L2.  The same
// kernel also runs one pass of one position per launch (with a separate
// select kernel in between) where the persistent launch is not available.
//
// Every wait gives up after two seconds: the kernel then records
// DSPARK_TIMEOUT in the workspace error word, lets the other roles of the CTA
// leave their loops, waits for its own TMA loads and stores, frees its TMEM
// and returns.  The other CTAs then give up at their next grid barrier.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <cstdlib>
#include <mutex>
#include <string>
#include <type_traits>

#include "common.cuh"
#include "draft_arith.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace dspark {
namespace tc {

constexpr int BM = 128;                              // rows per tile (TMEM lanes)
constexpr int BN = 192;                              // vocabulary columns per tile
constexpr int CW = 64;                               // columns per swizzle atom / chunk
constexpr int NCH = BN / CW;                         // chunks per tile
constexpr int KC = 64;                               // W2 rows per K-chunk
constexpr int kGroups = NCH;                         // epilogue groups: group g owns chunk g of every tile
constexpr int kEpiWarps = kGroups * 4;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;           // producer, MMA, epilogue
constexpr int kEpiWarp0 = 2;
constexpr int kStagingPerWarp = 32 * 32 * 4;         // [32 rows x 32 cols] fp32
constexpr uint32_t kW2Stage = KC * BN * 2;           // 24 KB
constexpr uint32_t kUChunk = BM * CW * 2;            // 16 KB: one 64-column chunk of U rows
constexpr uint32_t kUStage = NCH * kUChunk;          // 48 KB: the U rows of one tile
constexpr int NW = 3;                                // W2 ring stages of the W2 region
// Pass 1 writes no p_d, so its W2 ring also takes the two 24 KB halves of the
// (then idle) p_d staging area: five stages, more than a tile of W2 in flight.
constexpr int NW_S = 5;
// U ring stages.  A stage holds a whole tile and every epilogue warp waits on
// every use of it, in order: a mbarrier parity wait is only sound when the
// waiter has seen the previous phase complete, which a ring of chunk-sized
// stages dealt round-robin to the three groups would not guarantee.
constexpr int NU = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol0 = 128;                   // accumulators after the E columns
constexpr int kTailBytes = 1024;                     // mbarriers, TMEM slot, flags, tile queue
constexpr int kTq = 16;                              // tile queue: producer -> MMA and epilogue
constexpr size_t kSmemBytes =
    1024 + NW * (size_t)kW2Stage + NU * (size_t)kUStage + (size_t)kEpiWarps * kStagingPerWarp + kTailBytes;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kGroups * BM * 16 <= kEpiWarps * kStagingPerWarp, "segment merge fits in the staging buffers");
static_assert((NW_S - NW) * kW2Stage <= (uint32_t)(kEpiWarps * kStagingPerWarp), "pass-1 W2 stages fit in the staging area");

struct Params {
  int B, G, V, r, H;
  int k_begin, k_end;  // positions of this launch
  int pass_only;       // 0 or 1: that pass of position k_begin only; -1: both passes of every position
  int ntiles, nparts, ctas_per_m, n_ctas;
  uint64_t seed;
  const __nv_bfloat16* W1;   // [V, r]
  const __nv_bfloat16* Erows;  // [B, r] rows of the bias product (RNN head), or null: W1[x_{k-1}]
  const __nv_bfloat16* w;    // [H + r] confidence weight (w_e = w + H)
  const float* zh;           // [B, G] w_h . h
  const int32_t* anchor;     // [B]
  const float* temp;         // [B]
  const uint32_t* req_id;    // [B]
  float2* rowstat;           // [B] (m, S) of the current position
  float4* sel;               // [B] crossing chunk, sum before it, target u S, hit
  int32_t* tokens;           // [B, G]
  float4* part;              // [B, nparts] per 64-column chunk
  float2* pd_stat;           // [B, G] (m, S) of every drawn row, or null
  float4* segpart;           // [B, kDraftMaxSeg] per CTA segment
  float* pd_tok;
  float* conf_logit;
  float* conf;
  unsigned* gbar;            // grid barrier counter, zero at launch
  unsigned* sched;           // [G, n_mtiles] pass-2 tile counters, zero at launch
  int n_mtiles;
  WsHeader* hdr;
};

// first vocabulary tile of segment j when ntiles tiles are split into nseg
__host__ __device__ __forceinline__ int seg_begin(int j, int ntiles, int nseg) {
  return (int)(((long long)j * ntiles) / nseg);
}

// W1 row of a token just chosen into L2: the next position gathers it
__device__ __forceinline__ void prefetch_row(const __nv_bfloat16* row, int r) {
  for (int o = 0; o < r * 2; o += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(row) + o));
}

// bar.sync is warp-aligned: every caller reconverges its warp first
__device__ __forceinline__ void epi_sync() {
  __syncwarp();
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier among the epilogue threads of every CTA (all CTAs are
// resident: cooperative launch, one CTA per SM).  Returns false when the wait
// gave up.
__device__ bool grid_barrier(const Params& p, unsigned target, volatile int* abort_flag, volatile int* s_ok,
                             int epi_tid) {
  epi_sync();
  if (epi_tid == 0) {
    int ok = *abort_flag ? 0 : 1;
    __threadfence();
    if (ok) atomicAdd(p.gbar, 1u);
    if (ok && ld_acquire(p.gbar) < target) {
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ld_acquire(p.gbar) < target) {
        if (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  epi_sync();
  return *s_ok != 0;
}

// The draw of row b at position k ([DSpark] 方法细节, 草稿采样; inverse CDF in
// token-id order with u = Philox(seed, req, k + 1, draw 0)), one warp per row.
// Level 1 combines the segment partials (one per CTA of the row's M-tile, in
// vocabulary order) into the row max m and sum S and finds the segment where
// the running sum first exceeds u S; level 2 walks that segment's 64-column
// chunk partials to the crossing chunk.  The pass-2 CTA that owns the chunk
// then walks its 64 values.  Where rounding leaves no crossing, the last
// segment / chunk with positive mass is taken and the walk takes its last
// token with positive weight.  Greedy rows: the argmax (lowest id on ties).
__device__ __noinline__ void select_row(const Params& p, int b, int k, int lane) {
  constexpr unsigned FULL = 0xffffffffu;
  const int nseg = p.ctas_per_m;
  const float4* SP = p.segpart + (size_t)b * kDraftMaxSeg;
  if (!(p.temp[b] > 0.f)) {
    float av = -INFINITY;
    int ai = INT_MAX;
    for (int j = lane; j < nseg; j += 32) {
      const float4 s = __ldcg(&SP[j]);
      argmax_merge(av, ai, s.z, __float_as_int(s.w));
    }
    warp_argmax(av, ai);
    if (lane == 0) {
      p.tokens[(size_t)b * p.G + k] = ai;
      if (ai >= 0 && ai < p.V) prefetch_row(p.W1 + (size_t)ai * p.r, p.r);  // E of position k + 1
      p.rowstat[b] = make_float2(0.f, 1.f);
      if (p.pd_stat) p.pd_stat[(size_t)b * p.G + k] = make_float2(0.f, 1.f);
      p.sel[b] = make_float4(__int_as_float(-1), 0.f, 0.f, __int_as_float(0));
    }
    return;
  }
  constexpr int MAXT = kDraftMaxSeg / 32;
  float sm_[MAXT], ss_[MAXT];
  float m = -INFINITY;
#pragma unroll
  for (int t = 0; t < MAXT; ++t) {
    const int j = t * 32 + lane;
    float4 s = make_float4(-INFINITY, 0.f, 0.f, 0.f);
    if (j < nseg) s = __ldcg(&SP[j]);
    sm_[t] = s.x;
    ss_[t] = s.y;
    m = fmaxf(m, s.x);
  }
  m = warp_max(m);
  // masses of the segments relative to m, and their running sums in order
  float q[MAXT], incl[MAXT], excl[MAXT];
  float carry = 0.f;
#pragma unroll
  for (int t = 0; t < MAXT; ++t) {
    const int j = t * 32 + lane;
    q[t] = (j < nseg) ? tile_mass(sm_[t], ss_[t], m) : 0.f;
    incl[t] = __fadd_rn(carry, warp_inclusive_scan(q[t]));
    const float up = __shfl_up_sync(FULL, incl[t], 1);
    excl[t] = lane == 0 ? carry : up;
    carry = __shfl_sync(FULL, incl[t], 31);
  }
  const float S = carry;
  const float u = philox_uniform(p.seed, p.req_id[b], (uint32_t)(k + 1), 0u);
  const float target = u * S;
  int js = -1, jlast = -1;
  float base = 0.f;
#pragma unroll
  for (int t = 0; t < MAXT; ++t) {
    const int j = t * 32 + lane;
    const unsigned bal = __ballot_sync(FULL, j < nseg && incl[t] > target);
    if (js < 0 && bal) {
      const int L = __ffs(bal) - 1;
      js = t * 32 + L;
      base = __shfl_sync(FULL, excl[t], L);
    }
    const unsigned bp = __ballot_sync(FULL, j < nseg && q[t] > 0.f);
    if (bp) jlast = t * 32 + 31 - __clz(bp);
  }
  bool hit = js >= 0;
  if (!hit) js = max(jlast, 0);
  // level 2: the chunks of segment js
  const int c_lo = seg_begin(js, p.ntiles, nseg) * NCH;
  const int c_hi = min(seg_begin(js + 1, p.ntiles, nseg) * NCH, p.nparts);
  const float4* P = p.part + (size_t)b * p.nparts;
  int cstar = -1, clast = -1;
  float cbase = 0.f, run = base;
  for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
    const int cc = c0 + lane;
    float qc = 0.f;
    if (cc < c_hi) {
      const float4 pc = __ldcg(&P[cc]);
      qc = tile_mass(pc.x, pc.y, m);
    }
    const float inc = __fadd_rn(run, warp_inclusive_scan(qc));
    const float up = __shfl_up_sync(FULL, inc, 1);
    const float ex = lane == 0 ? run : up;
    if (hit && cstar < 0) {
      const unsigned bal = __ballot_sync(FULL, cc < c_hi && inc > target);
      if (bal) {
        const int L = __ffs(bal) - 1;
        cstar = c0 + L;
        cbase = __shfl_sync(FULL, ex, L);
      }
    }
    const unsigned bp = __ballot_sync(FULL, cc < c_hi && qc > 0.f);
    if (bp) clast = c0 + 31 - __clz(bp);
    run = __shfl_sync(FULL, inc, 31);
  }
  if (cstar < 0) {
    hit = false;
    cstar = clast >= 0 ? clast : c_lo;
  }
  if (lane == 0) {
    p.rowstat[b] = make_float2(m, S);
    if (p.pd_stat) p.pd_stat[(size_t)b * p.G + k] = make_float2(m, S);
    p.sel[b] = make_float4(__int_as_float(cstar), cbase, target, __int_as_float(hit ? 1 : 0));
  }
}

__global__ void __launch_bounds__(256) k_select_seg(Params p, int k) {
  const int b = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (b < p.B) select_row(p, b, k, threadIdx.x & 31);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_draft_tc(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmW2,
               const __grid_constant__ CUtensorMap tmPd, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int r = p.r;
  const int nkc = r / KC;  // K-chunks per tile
  uint8_t* sW = smem;
  uint8_t* sU = sW + NW * kW2Stage;
  uint8_t* sStg = sU + NU * kUStage;
  auto w2_slot = [&](int s) { return s < NW ? sW + s * kW2Stage : sStg + (s - NW) * kW2Stage; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + kEpiWarps * kStagingPerWarp);
  uint64_t* fullW = bars;
  uint64_t* emptyW = fullW + NW_S;
  uint64_t* fullU = emptyW + NW_S;
  uint64_t* emptyU = fullU + NU;
  uint64_t* tfull = emptyU + NU;
  uint64_t* tempty = tfull + 2;
  uint64_t* eready = tempty + 2;
  uint64_t* mma_done = eready + 1;
  uint64_t* stg_free = mma_done + 1;  // the epilogue's stores of a pass 2 have read the staging area
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stg_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = abort_flag + 1;
  // vocabulary tile of each item the producer hands on, in order; -1 ends a pass
  volatile int* tq = s_ok + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = (int)blockIdx.x / p.ctas_per_m;
  const int n_lo = (int)blockIdx.x % p.ctas_per_m;
  const int t_begin = seg_begin(n_lo, p.ntiles, p.ctas_per_m);
  const int count = seg_begin(n_lo + 1, p.ntiles, p.ctas_per_m) - t_begin;
  const int row_base = m_tile * BM;
  const bool persist = p.pass_only < 0;
  const int npass = persist ? 2 : 1;
  auto pass_of = [&](int pi) { return persist ? pi : p.pass_only; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NW_S; ++s) {
      ptx::mbar_init(&fullW[s], 1);
      ptx::mbar_init(&emptyW[s], 1);
    }
    for (int s = 0; s < NU; ++s) {
      ptx::mbar_init(&fullU[s], 1);
      ptx::mbar_init(&emptyU[s], kEpiWarps);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 2);  // the MMA commit and the issuing thread's own arrive
      ptx::mbar_init(&tempty[a], kEpiWarps);
    }
    ptx::mbar_init(eready, kEpiWarps);
    ptx::mbar_init(mma_done, 1);
    ptx::mbar_init(stg_free, kEpiWarps);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    report_error(p.hdr, DSPARK_TIMEOUT, (int)blockIdx.x);
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      const uint64_t pol_last = ptx::policy_evict_last();
      const uint64_t pol_first = ptx::policy_evict_first();
      int iu = 0, jt = 0;            // U stages, tile queue items
      uint32_t wpar = 0, wused = 0;  // per W2 slot: parity of its uses so far; used at all
      bool ok = true;
      for (int k = p.k_begin; k < p.k_end && ok; ++k)
        for (int pi = 0; pi < npass && ok; ++pi) {
          const int wr = pass_of(pi);
          const int nsl = wr == 0 ? NW_S : NW;
          int cs = 0;  // each pass cycles its W2 slots from slot 0
          // pass 1 after a pass 2 of this launch: its two extra slots are the
          // staging area, free once every epilogue warp's stores have read it
          bool stg_ok = !(wr == 0 && persist && k > p.k_begin);
          auto take_slot = [&](int& s) -> bool {
            s = cs;
            cs = cs + 1 == nsl ? 0 : cs + 1;
            if (s >= NW && !stg_ok) {
              if (!ptx::mbar_wait(stg_free, (uint32_t)((k - 1 - p.k_begin) & 1), abort_flag, kWaitLimitNs))
                return false;
              stg_ok = true;
            }
            const bool r = ptx::mbar_wait(&emptyW[s], ((wpar >> s) & 1) ^ 1, abort_flag, kWaitLimitNs);
            wpar ^= 1u << s;
            wused |= 1u << s;
            return r;
          };
          for (int i = 0; ok; ++i) {
            // the next tile: pass 1 walks this CTA's segment upward (the select
            // needs one partial per contiguous segment); pass 2 takes the M-tile's
            // tiles from a shared counter, top down, so that CTAs that run ahead
            // take more of them
            int n = -1;
            if (wr == 0) {
              if (i < count) n = t_begin + i;
            } else {
              const unsigned t = atomicAdd(&p.sched[(size_t)k * p.n_mtiles + m_tile], 1u);
              if (t < (unsigned)p.ntiles) n = p.ntiles - 1 - (int)t;
            }
            int s0;
            if (!take_slot(s0)) {
              ok = false;
              break;
            }
            tq[jt % kTq] = n;
            ++jt;
            if (n < 0) {
              // end of the pass: a W2 slot that carries no data
              ptx::mbar_arrive(&fullW[s0]);
              break;
            }
            const int v0 = n * BN;
            for (int kc = 0; kc < nkc; ++kc) {
              int s = s0;
              if (kc > 0 && !take_slot(s)) {
                ok = false;
                break;
              }
              uint8_t* st = w2_slot(s);
              ptx::mbar_expect_tx(&fullW[s], kW2Stage);
              for (int c = 0; c < NCH; ++c)
                ptx::tma_load_2d(st + c * (KC * CW * 2), &tmW2, &fullW[s], v0 + c * CW, kc * KC, pol_last);
            }
            if (ok) {
              const int s = iu % NU;
              if (!ptx::mbar_wait(&emptyU[s], ((iu / NU) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
              }
              ptx::mbar_expect_tx(&fullU[s], kUStage);
              for (int c = 0; c < NCH; ++c)
                ptx::tma_load_3d(sU + s * kUStage + c * kUChunk, &tmU, &fullU[s], v0 + c * CW, k, row_base,
                                 pol_first);
              ++iu;
            }
          }
        }
      if (!ok) fail();
      // every load this thread issued has landed before the CTA may exit: the
      // last use of each W2 slot and of each U stage
      for (int s = 0; s < NW_S; ++s)
        if ((wused >> s) & 1) ptx::mbar_wait(&fullW[s], ((wpar >> s) & 1) ^ 1, abort_flag, kWaitLimitNs);
      for (int j = max(0, iu - NU); j < iu; ++j) ptx::mbar_wait(&fullU[j % NU], (j / NU) & 1, abort_flag, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, false, true);
      int it = 0, jt = 0;  // accumulator uses, tile queue items
      uint32_t fpar = 0;   // per W2 slot: parity of its uses so far
      bool ok = true;
      for (int k = p.k_begin; k < p.k_end && ok; ++k) {
        // E of this position is in TMEM
        if (!ptx::mbar_wait(eready, (uint32_t)((k - p.k_begin) & 1), abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (int pi = 0; pi < npass && ok; ++pi) {
          const int nsl = pass_of(pi) == 0 ? NW_S : NW;
          int cs = 0;  // the producer's slot order
          auto next_slot = [&](int& s) -> bool {
            s = cs;
            cs = cs + 1 == nsl ? 0 : cs + 1;
            const bool r = ptx::mbar_wait(&fullW[s], (fpar >> s) & 1, abort_flag, kWaitLimitNs);
            fpar ^= 1u << s;
            return r;
          };
          for (;;) {
            const int a = it & 1;
            int s0;
            if (!ptx::mbar_wait(&tempty[a], ((it >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs) || !next_slot(s0)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const int n = tq[jt % kTq];
            ++jt;
            ++it;
            if (n < 0) {
              // end of the pass: release the empty W2 slot and hand the marker on
              ptx::mbar_arrive(&emptyW[s0]);
              ptx::mbar_arrive(&tfull[a]);
              ptx::mbar_arrive(&tfull[a]);
              break;
            }
            const uint32_t d = tmem + kAccCol0 + (uint32_t)(a * BN);
            for (int kc = 0; kc < nkc; ++kc) {
              int s = s0;
              if (kc > 0) {
                if (!next_slot(s)) {
                  ok = false;
                  break;
                }
                ptx::tc_fence_after();
              }
              const uint32_t aW2 = ptx::smem_u32(w2_slot(s));
#pragma unroll
              for (int k4 = 0; k4 < KC / 16; ++k4) {
                const int ks = kc * (KC / 16) + k4;
                // B: W2 K-chunk [64 x 192], MN-major, 128B swizzle: three 64-column
                //    blocks of 64 rows x 128 B, 8 KB apart (leading offset); 8-row
                //    groups 1024 B apart along K (stride offset); a K step of 16 is
                //    two groups
                const uint64_t bd = ptx::smem_desc_sw128(aW2 + k4 * 2048, KC * CW * 2, 1024);
                // A: E in TMEM, a K step of 16 bf16 = 8 columns
                ptx::tc_mma_tmem_a(d, tmem + (uint32_t)(ks * 8), bd, idesc, ks > 0 ? 1u : 0u);
              }
              ptx::tc_commit(&emptyW[s]);
            }
            if (!ok) break;
            ptx::tc_commit(&tfull[a]);
            // this thread's own arrive orders its reads of the tile queue
            // before the epilogue's
            ptx::mbar_arrive(&tfull[a]);
          }
        }
      }
      if (!ok) fail();
      // TMEM is not freed under a running MMA
      ptx::tc_commit(mma_done);
      ptx::mbar_wait(mma_done, 0, abort_flag, kWaitLimitNs);
    }
  } else {
    // ------------------------------ epilogue ----------------------------------
    const int ew = warp - kEpiWarp0;        // epilogue warp 0..11
    const int epi_tid = ew * 32 + lane;
    const int g = ew >> 2;                  // group: chunk g of every tile
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;          // row within the M-tile
    const int b = row_base + row;
    const bool vrow = b < p.B;
    const uint32_t lane_bits = (uint32_t)(q * 32) << 16;
    const int npieces = r / 64;  // 64-element pieces of an E row (32 TMEM columns each)
    const float T_ = vrow ? p.temp[b] : 1.f;
    const bool sampled = T_ > 0.f;
    const float c = row_scale(T_);
    uint8_t* stg = sStg + ew * kStagingPerWarp;
    unsigned nbar = 0;  // grid barriers passed
    int it = 0;         // accumulator uses (tiles and end markers)
    int jt = 0;         // tile queue items
    int nut = 0;        // tiles consumed (U ring uses)
    // cleared only by a failed grid barrier, whose outcome every epilogue warp
    // of the CTA reads from shared memory: the warps leave together
    bool alive = true;

    for (int k = p.k_begin; k < p.k_end && alive; ++k) {
      {
        // E = W1[x_{k-1}] (x_0 = anchor) into TMEM columns [0, r/2): two bf16
        // per column, zeros past B.  Group g copies the 64-element pieces g and
        // g + 3 of its rows.
        int x = 0;
        if (vrow) {
          x = (k == 0) ? p.anchor[b] : __ldcg(&p.tokens[(size_t)b * p.G + k - 1]);
          if (x < 0 || x >= p.V) {
            if (g == 0) report_error(p.hdr, DSPARK_BAD_INPUT, x);
            x = 0;
          }
        }
        const uint4* src = reinterpret_cast<const uint4*>(p.Erows ? p.Erows + (size_t)(vrow ? b : 0) * r
                                                                  : p.W1 + (size_t)x * r);
        // one 32-column piece at a time keeps the gather within the register
        // budget; the token's writer prefetched the row into L2
#pragma unroll 1
        for (int s = 0; s < 2; ++s) {
          const int pc = g + kGroups * s;
          if (pc < npieces) {
            uint32_t wv[32];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint4 qv = vrow ? src[pc * 8 + e] : make_uint4(0u, 0u, 0u, 0u);
              wv[4 * e] = qv.x;
              wv[4 * e + 1] = qv.y;
              wv[4 * e + 2] = qv.z;
              wv[4 * e + 3] = qv.w;
            }
            __syncwarp();  // tcgen05.st is warp-collective
            ptx::tmem_st32(tmem + lane_bits + (uint32_t)(pc * 32), wv);
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(eready);
      }
      if (pass_of(0) == 0 && g == 0 && n_lo == 0 && !p.Erows) {
        // the first CTA of the M-tile also forms the confidence of position k:
        // z = w_h . h_k + w_e . W1[x_{k-1}], reading the E row back from TMEM
        // once every group has stored its pieces
        const bool ok = ptx::mbar_wait(eready, (uint32_t)((k - p.k_begin) & 1), abort_flag, kWaitLimitNs);
        if (__all_sync(0xffffffffu, ok)) {
          ptx::tc_fence_after();
          const uint4* wsrc = reinterpret_cast<const uint4*>(p.w + p.H);
          float zacc = 0.f;
          for (int pc = 0; pc < npieces; ++pc) {
            float ev[32];  // bf16 pairs, as raw bits
            ptx::tmem_ld32(tmem + lane_bits + (uint32_t)(pc * 32), ev);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint4 we = wsrc[pc * 8 + e];
              const uint32_t wq[4] = {we.x, we.y, we.z, we.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const uint32_t eb = __float_as_uint(ev[4 * e + t]);
                const float2 fe = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&eb));
                const float2 fw = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wq[t]));
                zacc = fmaf(fw.x, fe.x, zacc);
                zacc = fmaf(fw.y, fe.y, zacc);
              }
            }
          }
          if (vrow) {
            const float z = p.zh[(size_t)b * p.G + k] + zacc;
            p.conf_logit[(size_t)b * p.G + k] = z;
            p.conf[(size_t)b * p.G + k] = 1.f / (1.f + expf(-z));
          }
        } else if (lane == 0) {
          fail();
        }
      }

      for (int pi = 0; pi < npass && alive; ++pi) {
        const int wr = pass_of(pi);
        // the pass body is instantiated once per pass, so that each keeps only
        // its own per-row state live across the tile loop
        auto run_pass = [&](auto wr_c) {
          constexpr int wr = decltype(wr_c)::value;
          // pass 2 row data: (m, 1/S), and the crossing chunk of sampled rows or
          // the token of greedy rows (written by the select)
          float rm = 0.f, rinvS = 1.f, sbase = 0.f, starget = 0.f;
          int xb = -1, cstar = -1;
          bool shit = false;
          if (wr == 1 && vrow) {
            const float2 st = __ldcg(&p.rowstat[b]);
            rm = st.x;
            rinvS = inv_sum(st.y);
            if (sampled) {
              const float4 sv = __ldcg(&p.sel[b]);
              cstar = __float_as_int(sv.x);
              sbase = sv.y;
              starget = sv.z;
              shit = __float_as_int(sv.w) != 0;
            } else {
              xb = __ldcg(&p.tokens[(size_t)b * p.G + k]);
            }
          }
          // pass 1: this group's running partial over its chunks of the segment
          float gm = -INFINITY, gs = 0.f, gav = -INFINITY;
          int gai = INT_MAX;
          float pdtok = 0.f;
          bool have_pdtok = false;
          const int ch = g;  // the chunk of every tile this group owns
          for (;;) {
            const int a = it & 1;
            bool ok = ptx::mbar_wait(&tfull[a], (it >> 1) & 1, abort_flag, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, ok)) {
              // leave the tile loop only: every warp still meets the named
              // barriers below, where the CTA decides together to stop
              if (lane == 0) fail();
              break;
            }
            ptx::tc_fence_after();
            const int n = tq[jt % kTq];
            ++jt;
            ++it;
            if (n < 0) {  // end of the pass
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(&tempty[a]);
              break;
            }
            const int v0 = n * BN + ch * CW;
            const int su = nut % NU;
            ok = ptx::mbar_wait(&fullU[su], (nut / NU) & 1, abort_flag, kWaitLimitNs);
            ++nut;
            if (!__all_sync(0xffffffffu, ok)) {
              if (lane == 0) fail();
              break;
            }
            const uint32_t ta = tmem + lane_bits + kAccCol0 + (uint32_t)(a * BN + ch * CW);
            const uint8_t* su_row = sU + su * kUStage + ch * kUChunk + row * 128;
            const int nvalid = min(CW, p.V - v0);  // columns past V are masked
            // The logits l of columns v0 + 32 h .. + 31: TMEM accumulator + U (4
            // of the row's 8 swizzled 16-byte chunks of 8 bf16).  The chunk is
            // handled in 32-column halves so that only 32 values are live; the
            // last read of the tile releases the accumulator and the U stage.
            auto load_half = [&](int h, float(&x)[32], bool last) {
              // tcgen05.ld is warp-collective: reconverge the lanes, which took
              // different branches for greedy and sampled rows, before it
              __syncwarp();
              ptx::tmem_ld32(ta + 32 * h, x);
              ptx::tmem_ld_wait();
              if (last) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&tempty[a]);
              }
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const int c8 = 4 * h + cc;
                const uint4 qv = *reinterpret_cast<const uint4*>(su_row + ((c8 ^ (row & 7)) << 4));
                const __nv_bfloat162* bp = reinterpret_cast<const __nv_bfloat162*>(&qv);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 f = __bfloat1622float2(bp[e]);
                  x[8 * cc + 2 * e] = add_base(f.x, x[8 * cc + 2 * e]);
                  x[8 * cc + 2 * e + 1] = add_base(f.y, x[8 * cc + 2 * e + 1]);
                }
              }
              if (last) {
                // the stage's next fill is an async-proxy (TMA) write: order
                // this warp's generic reads before it
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&emptyU[su]);
              }
            };
            if constexpr (wr == 0) {
              // sampled rows: y = l c, the chunk's max and sum of 2^(y - max),
              // each 32-column half reduced on its own and merged; greedy rows:
              // the argmax of l, ties to the lowest column
              float mc = -INFINITY, cs = 0.f, av = -INFINITY;
              int ai = INT_MAX;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float x[32];
                load_half(h, x, h == 1);
                if (sampled) {
                  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                  for (int j = 0; j < 32; ++j) {
                    x[j] = (32 * h + j < nvalid) ? scale_logit(x[j], c) : -INFINITY;
                    mx[j & 3] = fmaxf(mx[j & 3], x[j]);
                  }
                  const float mh = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                  if (mh != -INFINITY) {
                    float sm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 32; ++j) sm[j & 3] += exp_shifted(x[j], mh);
                    const float sh = (sm[0] + sm[1]) + (sm[2] + sm[3]);
                    const float nm = fmaxf(mc, mh);
                    cs = __fadd_rn(tile_mass(mc, cs, nm), tile_mass(mh, sh, nm));
                    mc = nm;
                  }
                } else {
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    if (32 * h + j < nvalid && x[j] > av) {
                      av = x[j];
                      ai = v0 + 32 * h + j;
                    }
                }
              }
              if (!sampled) {
                mc = av;
                cs = 1.f;
              }
              if (v0 < p.V) {
                // one partial per 64-column chunk: (max y, sum 2^(y - max), argmax)
                if (vrow) p.part[(size_t)b * p.nparts + v0 / CW] = make_float4(mc, cs, av, __int_as_float(ai));
                const float nm = fmaxf(gm, mc);
                gs = __fadd_rn(tile_mass(gm, gs, nm), tile_mass(mc, cs, nm));
                gm = nm;
                argmax_merge(gav, gai, av, ai);
              }
            } else {
              // numerators w = 2^(y - m) (sampled rows) and p = w / S; the draw:
              // the select named the chunk where the prefix sum of w crosses u S
              // and the sum before it; the thread walks that chunk in token order
              // with exactly the values it writes.  Rounding that leaves no
              // crossing picks the chunk's last token with positive weight.
              const bool walk = v0 / CW == cstar;
              float run = sbase, pf = 0.f, pl = 0.f;
              int xf = -1, xl = -1;
              const int row0 = row_base + q * 32;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float x[32];
                load_half(h, x, h == 1);
                if (sampled) {
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    x[j] = (32 * h + j < nvalid) ? exp_shifted(scale_logit(x[j], c), rm) : 0.f;
                }
                if (walk) {
#pragma unroll
                  for (int j = 0; j < 32; ++j) {
                    const float wj = x[j];
                    if (wj > 0.f) {
                      xl = v0 + 32 * h + j;
                      pl = wj;
                    }
                    run += wj;
                    if (xf < 0 && shit && run > starget) {
                      xf = v0 + 32 * h + j;
                      pf = wj;
                    }
                  }
                }
                // the previous TMA store must have read the staging buffer
                if (lane == 0) ptx::bulk_wait_read0();
                __syncwarp();
                if (sampled) {
#pragma unroll
                  for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<float4*>(stg + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                        make_float4(__fmul_rn(x[4 * cc], rinvS), __fmul_rn(x[4 * cc + 1], rinvS),
                                    __fmul_rn(x[4 * cc + 2], rinvS), __fmul_rn(x[4 * cc + 3], rinvS));
                } else {
                  // greedy rows: the one-hot row of the chosen token
                  const int jx = xb - (v0 + 32 * h);
#pragma unroll
                  for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<float4*>(stg + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                        make_float4(jx == 4 * cc ? 1.f : 0.f, jx == 4 * cc + 1 ? 1.f : 0.f,
                                    jx == 4 * cc + 2 ? 1.f : 0.f, jx == 4 * cc + 3 ? 1.f : 0.f);
                  if (jx >= 0 && jx < 32) {
                    pdtok = 1.f;
                    have_pdtok = true;
                  }
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 < p.B && v0 + 32 * h < p.V) {  // boxes that start past B or V would write nothing
                  // p_d is streamed out once: evict-first
                  ptx::tma_store_3d(&tmPd, stg, v0 + 32 * h, k, row0, ptx::policy_evict_first());
                  ptx::bulk_commit();
                }
              }
              if (walk) {
                if (xf < 0) {
                  xf = xl;
                  pf = pl;
                }
                if (xf >= 0) {
                  p.tokens[(size_t)b * p.G + k] = xf;
                  prefetch_row(p.W1 + (size_t)xf * r, r);  // E of position k + 1
                  pdtok = __fmul_rn(pf, rinvS);
                  have_pdtok = true;
                }
              }
            }
          }
          if constexpr (wr == 0) {
            // segment partial of each row: merge the three groups' running
            // partials through the (idle) staging buffers
            if (lane == 0) ptx::bulk_wait_read0();
            __syncwarp();
            float4* xch = reinterpret_cast<float4*>(sStg);
            epi_sync();
            xch[g * BM + row] = make_float4(gm, gs, gav, __int_as_float(gai));
            epi_sync();
            if (g == 0 && vrow && !*abort_flag) {
              float m = gm;
              for (int gg = 1; gg < kGroups; ++gg) m = fmaxf(m, xch[gg * BM + row].x);
              float s = 0.f, av = -INFINITY;
              int ai = INT_MAX;
              for (int gg = 0; gg < kGroups; ++gg) {
                const float4 e = xch[gg * BM + row];
                if (m != -INFINITY) s = __fadd_rn(s, tile_mass(e.x, e.y, m));
                argmax_merge(av, ai, e.z, __float_as_int(e.w));
              }
              p.segpart[(size_t)b * kDraftMaxSeg + n_lo] = make_float4(m, s, av, __int_as_float(ai));
            }
          } else {
            if (vrow && have_pdtok && !*abort_flag) p.pd_tok[(size_t)b * p.G + k] = pdtok;
            // this warp's stores have read the staging area: the next pass 1 may
            // load W2 into it
            if (lane == 0) ptx::bulk_wait_read0();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(stg_free);
          }
        };
        if (wr == 0)
          run_pass(std::integral_constant<int, 0>{});
        else
          run_pass(std::integral_constant<int, 1>{});
        if (wr == 0) {
          if (persist) {
            if (!grid_barrier(p, ++nbar * (unsigned)p.n_ctas, abort_flag, s_ok, epi_tid)) {
              if (epi_tid == 0) fail();
              alive = false;
              break;
            }
            for (int rb = (int)blockIdx.x + p.n_ctas * ew; rb < p.B; rb += p.n_ctas * kEpiWarps)
              select_row(p, rb, k, lane);
            if (!grid_barrier(p, ++nbar * (unsigned)p.n_ctas, abort_flag, s_ok, epi_tid)) {
              if (epi_tid == 0) fail();
              alive = false;
              break;
            }
          }
        } else if (persist && k + 1 < p.k_end) {
          // every token of position k is written before E of k + 1 is gathered
          if (!grid_barrier(p, ++nbar * (unsigned)p.n_ctas, abort_flag, s_ok, epi_tid)) {
            if (epi_tid == 0) fail();
            alive = false;
            break;
          }
        }
      }
    }
    if (lane == 0) ptx::bulk_wait0();
  }

  // lanes 1-31 of the producer and MMA warps wait here for lane 0: reconverge
  // every warp before the CTA-wide barrier
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

static bool encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DevInfo {
  int sms = 0;
  bool sm103 = false;
  bool coop = false;
};

static DevInfo dev_info() {
  static DevInfo cache[64];
  static bool have[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DevInfo{};
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    int major = 0, minor = 0, sms = 0, coop = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    cache[dev].sms = sms;
    cache[dev].sm103 = (major == 10 && minor == 3);
    cache[dev].coop = coop != 0;
    have[dev] = true;
  }
  return cache[dev];
}

// DSPARK_DRAFT_LAUNCH=per_pass: one launch per pass and a select kernel in
// between instead of the persistent launch (the tests use it to cover both)
static bool per_pass_forced() {
  static bool forced = false;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* e = getenv("DSPARK_DRAFT_LAUNCH");
    forced = e && std::string(e) == "per_pass";
  });
  return forced;
}

}  // namespace tc

// Which logits path the draft sampler uses: tensor cores when the shape fits
// the tile (bf16, r a multiple of 64 up to 256, V a multiple of 8) on an
// sm_103 device; otherwise the CUDA-core path.  DSPARK_DRAFT_PATH=cuda_core
// forces the CUDA-core path (used by the tests to cover both paths).
// ---------------------------------------------------------------------------
// RNN head: P [B gamma, 3r] = h [B gamma, H] . W_rnn[:, 2r:]^T on the tensor cores
// ([DSpark] 方法细节, "RNN头的实现": the h_k part of W z_k does not depend on the
// recurrence, so every position's share is one bf16 GEMM with fp32
// accumulation).  128 x 128 tiles, K in 64-element chunks through a ring of
// four stages (A and B both K-major, 128B-swizzled by TMA), the accumulator in
// 128 TMEM columns.  Warp 0 loads, warp 1 issues the MMAs, all four warps
// read TMEM lane quarters and store fp32 rows.  Every wait is bounded.
// ---------------------------------------------------------------------------
namespace hp {
constexpr int TM = 128, TN = 128, TK = 64, NS = 4;
constexpr uint32_t kTileBytes = TM * TK * 2;  // 16 KB, A and B tiles alike
constexpr uint32_t kSmem = NS * 2 * kTileBytes + 1024;
}  // namespace hp

__global__ void __launch_bounds__(128, 1) k_rnn_hproj_tc(const __grid_constant__ CUtensorMap tmA,
                                                        const __grid_constant__ CUtensorMap tmB, float* P, int M,
                                                        int N, int K, WsHeader* hdr) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[hp::NS], empty[hp::NS], done;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * hp::TM, n0 = blockIdx.x * hp::TN;
  const int nk = (K + hp::TK - 1) / hp::TK;
  volatile int* abort_flag = &abort_s;
  if (threadIdx.x == 0) {
    for (int i = 0; i < hp::NS; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(&done, 1);
    ptx::fence_mbar_init();
    abort_s = 0;
  }
  if (warp == 1) {
    ptx::tmem_alloc(&tmem_slot, 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  auto fail = [&]() {
    if (hdr) report_error(hdr, DSPARK_TIMEOUT, (int)blockIdx.x);
    *abort_flag = 1;
  };
  if (warp == 0 && lane == 0) {
    const uint64_t pol = ptx::policy_evict_last();
    for (int kc = 0; kc < nk && !*abort_flag; ++kc) {
      const int st = kc % hp::NS;
      if (kc >= hp::NS && !ptx::mbar_wait(&empty[st], ((kc / hp::NS) - 1) & 1, abort_flag, tc::kWaitLimitNs)) {
        fail();
        break;
      }
      uint8_t* a = sm + st * 2 * hp::kTileBytes;
      ptx::mbar_expect_tx(&full[st], 2 * hp::kTileBytes);
      ptx::tma_load_2d(a, &tmA, &full[st], kc * hp::TK, m0, pol);
      ptx::tma_load_2d(a + hp::kTileBytes, &tmB, &full[st], kc * hp::TK, n0, pol);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(hp::TM, hp::TN, false, false);
    bool ok = true;
    for (int kc = 0; kc < nk && ok; ++kc) {
      const int st = kc % hp::NS;
      if (!ptx::mbar_wait(&full[st], (kc / hp::NS) & 1, abort_flag, tc::kWaitLimitNs)) {
        fail();
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t a = ptx::smem_u32(sm + st * 2 * hp::kTileBytes);
#pragma unroll
      for (int kk = 0; kk < hp::TK / 16; ++kk) {
        // K-major, 128B swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart;
        // the 16-element K step is 32 bytes inside the atom
        const uint64_t ad = ptx::smem_desc_sw128(a + kk * 32, 16, 1024);
        const uint64_t bd = ptx::smem_desc_sw128(a + hp::kTileBytes + kk * 32, 16, 1024);
        ptx::tc_mma(tmem, ad, bd, idesc, (kc | kk) ? 1u : 0u);
      }
      ptx::tc_commit(&empty[st]);
    }
    ptx::tc_commit(&done);
  }
  __syncwarp();
  // epilogue: TMEM lane quarter of this warp, 128 columns in four loads
  const bool ok = ptx::mbar_wait(&done, 0, abort_flag, tc::kWaitLimitNs);
  if (__all_sync(0xffffffffu, ok)) {
    ptx::tc_fence_after();
    const int row = m0 + warp * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < hp::TN / 32; ++c) {
      float v[32];
      ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c * 32), v);
      ptx::tmem_ld_wait();
      if (row < M) {
        float* dst = P + (size_t)row * N + n0 + c * 32;
        const int nv = min(32, N - (n0 + c * 32));
        if (nv == 32 && (((uintptr_t)dst) & 15) == 0) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q)
            if (q < nv) dst[q] = v[q];
        }
      }
    }
  } else if (lane == 0) {
    fail();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) ptx::tmem_dealloc(tmem, 128);
}

bool rnn_hproj_tc_supported(const dspark_dims& d) {
  return d.dtype == DSPARK_BF16 && d.H >= 8 && (d.H % 8) == 0 && (d.r % 8) == 0 && tc::dev_info().sm103 &&
         tc::encode_fn() != nullptr;
}

// C[M, N] (fp32, row stride N) = A[M, K] . B[N, K]^T for bf16 A and B with K
// contiguous (row strides lda, ldb elements, multiples of 8; 16-byte aligned
// bases): the k_rnn_hproj_tc tiles, K-major operands by TMA.
cudaError_t launch_tc_gemm_nt(const void* A, int lda, const void* Bm, int ldb, float* C, int M, int N, int K,
                              WsHeader* hdr, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)lda * 2};
    const cuuint32_t box[2] = {hp::TK, hp::TM};
    if (!tc::encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)ldb * 2};
    const cuuint32_t box[2] = {hp::TK, hp::TN};
    if (!tc::encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Bm, dims, strides, box)) return cudaErrorInvalidValue;
  }
  if (const cudaError_t ae = ensure_smem_limit((const void*)k_rnn_hproj_tc, (int)hp::kSmem); ae != cudaSuccess)
    return ae;
  const dim3 grid((N + hp::TN - 1) / hp::TN, (M + hp::TM - 1) / hp::TM);
  k_rnn_hproj_tc<<<grid, 128, hp::kSmem, s>>>(tmA, tmB, C, M, N, K, hdr);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_rnn_hproj_tc(const dspark_draft_args& a, float* P, WsHeader* hdr, cudaStream_t s) {
  const dspark_dims& d = a.dims;
  // h [B gamma, H] . W_rnn[:, 2r:]^T (rows of stride 2r + H)
  return launch_tc_gemm_nt(a.h, d.H, static_cast<const __nv_bfloat16*>(a.W_rnn) + 2 * d.r, 2 * d.r + d.H, P,
                           d.B * d.gamma, 3 * d.r, d.H, hdr, s);
}

bool draft_tc_supported(const dspark_dims& d) {
  static int forced = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* e = getenv("DSPARK_DRAFT_PATH");
    forced = (e && std::string(e) == "cuda_core") ? 0 : 1;
  });
  if (!forced) return false;
  if (d.dtype != DSPARK_BF16 || d.r < 64 || d.r > 256 || (d.r % 64) != 0 || (d.V % 8) != 0 || (d.H % 8) != 0)
    return false;
  return tc::dev_info().sm103 && tc::encode_fn() != nullptr;
}

cudaError_t launch_draft_tc(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s,
                            const std::function<cudaError_t(int)>* hook, const void* Erows) {
  const dspark_dims& d = a.dims;
  const cuuint64_t V = (cuuint64_t)d.V, G = (cuuint64_t)d.gamma, B = (cuuint64_t)d.B, r = (cuuint64_t)d.r;
  CUtensorMap tmU, tmW2, tmPd;
  {  // U [B, G, V] bf16 as (v, k, b)
    const cuuint64_t dims[3] = {V, G, B};
    const cuuint64_t strides[2] = {V * 2, G * V * 2};
    const cuuint32_t box[3] = {tc::CW, 1, tc::BM};
    if (!tc::encode(&tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.U, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {  // W2 [r, V] bf16 as (v, i)
    const cuuint64_t dims[2] = {V, r};
    const cuuint64_t strides[1] = {V * 2};
    const cuuint32_t box[2] = {tc::CW, tc::KC};
    if (!tc::encode(&tmW2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {  // p_d rows [B, G, V] fp32 as (v, k, b); stores of 32 columns x 32 rows
    const cuuint64_t dims[3] = {V, G, B};
    const cuuint64_t strides[2] = {V * 4, G * V * 4};
    const cuuint32_t box[3] = {32, 1, 32};
    if (!tc::encode(&tmPd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.pd_rows, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  if (const cudaError_t ae = ensure_smem_limit((const void*)tc::k_draft_tc, (int)tc::kSmemBytes); ae != cudaSuccess)
    return ae;

  tc::Params p;
  p.B = d.B;
  p.G = d.gamma;
  p.V = d.V;
  p.r = d.r;
  p.H = d.H;
  p.seed = a.seed;
  p.ntiles = (d.V + tc::BN - 1) / tc::BN;
  p.nparts = (d.V + tc::CW - 1) / tc::CW;
  const int n_mtiles = (d.B + tc::BM - 1) / tc::BM;
  const tc::DevInfo di = tc::dev_info();
  const int sms = di.sms > 0 ? di.sms : 148;
  p.ctas_per_m = std::max(1, std::min(std::min(p.ntiles, sms / n_mtiles), kDraftMaxSeg));
  p.n_ctas = n_mtiles * p.ctas_per_m;
  p.W1 = static_cast<const __nv_bfloat16*>(a.W1);
  p.Erows = static_cast<const __nv_bfloat16*>(Erows);
  p.w = static_cast<const __nv_bfloat16*>(a.w);
  p.zh = reinterpret_cast<const float*>(ws + L.zh);
  p.anchor = a.anchor;
  p.temp = a.temp;
  p.req_id = a.req_id;
  p.rowstat = reinterpret_cast<float2*>(ws + L.rowstat);
  p.sel = reinterpret_cast<float4*>(ws + L.sel);
  p.tokens = a.tokens;
  p.part = reinterpret_cast<float4*>(ws + L.part);
  p.pd_stat = reinterpret_cast<float2*>(a.pd_stat);
  p.segpart = reinterpret_cast<float4*>(ws + L.segpart);
  p.pd_tok = a.pd_tok;
  p.conf_logit = a.conf_logit;
  p.conf = a.conf;
  p.gbar = reinterpret_cast<unsigned*>(ws + L.gbar);
  p.sched = reinterpret_cast<unsigned*>(ws + L.gbar + 16);
  p.n_mtiles = n_mtiles;
  const size_t sync_bytes = 16 + (size_t)d.gamma * n_mtiles * sizeof(unsigned);
  p.hdr = reinterpret_cast<WsHeader*>(ws);

  // Persistent launch: all CTAs resident (one per SM), so the grid barriers
  // inside are safe; the cooperative attribute makes the launch fail rather
  // than run with CTAs waiting for an SM.
  cudaError_t e = cudaMemsetAsync(p.gbar, 0, sync_bytes, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_ctas);
  cfg.blockDim = dim3(tc::kThreads);
  cfg.dynamicSmemBytes = tc::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!tc::per_pass_forced() && di.coop && n_mtiles <= sms) {
    if (!hook) {
      p.k_begin = 0;
      p.k_end = d.gamma;
      p.pass_only = -1;
      count_launches(1);
      return cudaLaunchKernelEx(&cfg, tc::k_draft_tc, tmU, tmW2, tmPd, p);
    }
    // with a hook: one persistent launch per position (both passes and the
    // select inside), the hook before it; the grid-barrier counter restarts
    // at zero for every launch, the pass-2 tile counters are per position
    p.pass_only = -1;
    for (int k = 0; k < d.gamma; ++k) {
      e = (*hook)(k);
      if (e == cudaSuccess && k > 0) e = cudaMemsetAsync(p.gbar, 0, 16, s);
      if (e != cudaSuccess) return e;
      p.k_begin = k;
      p.k_end = k + 1;
      e = cudaLaunchKernelEx(&cfg, tc::k_draft_tc, tmU, tmW2, tmPd, p);
      if (e != cudaSuccess) return e;
    }
    count_launches(d.gamma);
    return cudaSuccess;
  }
  count_launches(3 * d.gamma);
  for (int k = 0; k < d.gamma; ++k) {
    if (hook) {
      e = (*hook)(k);
      if (e != cudaSuccess) return e;
    }
    p.k_begin = k;
    p.k_end = k + 1;
    p.pass_only = 0;
    tc::k_draft_tc<<<p.n_ctas, tc::kThreads, tc::kSmemBytes, s>>>(tmU, tmW2, tmPd, p);
    tc::k_select_seg<<<(d.B + 7) / 8, 256, 0, s>>>(p, k);
    p.pass_only = 1;
    tc::k_draft_tc<<<p.n_ctas, tc::kThreads, tc::kSmemBytes, s>>>(tmU, tmW2, tmPd, p);
  }
  return cudaGetLastError();
}

}  // namespace dspark
