// Fused-sweep tensor-core draft sampler, sm_103a: the Markov head, and the
// RNN head, whose recurrent step runs in each gather (rnn_units below).
//
// Position k of the draft needs two passes over the vocabulary: one for the
// row normaliser of p_d^k, one that writes p_d^k ([DSpark] 方法细节, "马尔可夫头
// （Markov head）的实现"; the logits of a position do not fit on chip).  The
// second pass of position k and the first pass of position k + 1 read the
// same W2 tiles, so this kernel runs them as ONE sweep: every W2 tile it
// loads serves two tcgen05.mma products,
//     W item  l = U_k     + E_k     . W2   -> p_d^k written (needs m_k, S_k)
//     S item  l = U_{k+1} + E_{k+1} . W2   -> (max, sum 2^(y - max), argmax)
//                                             partials of position k + 1
// which halves the W2 traffic of the two-pass scheme.  The sweep needs E_{k+1}
// = W1[x_k] at its start, so the token x_k is chosen before it: the select,
// from the chunk partials of the previous sweep, finds the 64-column chunk
// where the inverse CDF crosses u S and recomputes that chunk's logits on the
// CUDA cores (the E_k . W2 dot products in fp32) to walk it.  One persistent
// cooperative launch runs all sweeps: S(0), then W(k) + S(k + 1) for
// k = 0 .. gamma - 1.  A grid barrier separates a sweep from its select; the
// next sweep waits only for the tokens of its own rows (release/acquire).
// The CTAs serving an M-tile claim its vocabulary tiles one by one, so that
// they finish a sweep together whatever their memory bandwidth.
//
// Tile 128 requests x 128 vocabulary columns.  TMEM: E_k and E_{k+1} in two
// slots of r/2 columns, then two 128-column fp32 accumulators.
//   warp 0    TMA producer: W2 K-chunks [64 x 128] (six stages), U tiles
//             [128 x 128] per item (three stages)
//   warp 1    tcgen05.mma issuer: per tile the W item then the S item on the
//             same W2 stages, alternating accumulators
//   warps 2-9 epilogue, two groups of four warps; group g owns the g-th
//             64-column chunk of every item.  They also gather E and run
//             the select (two teams of four warps, one row each).
// For B <= 16, k_draft_narrow (below) puts the vocabulary on the MMA's M side
// instead, with the requests as N = 16 columns.
// Every wait gives up after two seconds and the kernel records DSPARK_TIMEOUT.
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
namespace fz {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int CW = 64;
constexpr int NCH = BN / CW;
constexpr int KC = 64;
constexpr int kGroups = NCH;
constexpr int kEpiWarps = kGroups * 4;
constexpr int kTeamWarps = kEpiWarps / 2;  // the select recomputes two rows at a time
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kEpiWarp0 = 2;
constexpr int kStagingPerWarp = 32 * 32 * 4;
constexpr uint32_t kW2Stage = KC * BN * 2;     // 16 KB
constexpr uint32_t kUChunk = BM * CW * 2;      // 16 KB
constexpr uint32_t kUStage = NCH * kUChunk;    // 32 KB: the U rows of one item
// Stage rings of the 128-row form, a template parameter of its kernel: the W2
// ring (16 KB stages, four per tile at r = 256) and the U ring (32 KB stages,
// one per item), in the shared memory the p_d staging leaves.  With few
// M-tiles every W2 tile comes from DRAM and the deeper W2 ring pays; with many,
// the M-tiles' CTAs find most W2 tiles in L2 and U (read from DRAM by every
// CTA) wants the deeper U ring.
constexpr int kRingW2Deep = 0;                 // 8 W2 stages (two tiles), 2 U stages
constexpr int kRingUDeep = 1;                  // 6 W2 stages (1.5 tiles), 3 U stages
__host__ __device__ constexpr int ring_nw(int ring) { return ring == kRingW2Deep ? 8 : 6; }
__host__ __device__ constexpr int ring_nu(int ring) { return ring == kRingW2Deep ? 2 : 3; }
constexpr int kRingW2DeepMaxMtiles = 4;        // M-tiles up to which the W2-deep ring runs (measured)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kESlotCols = 128;           // r / 2 columns, r <= 256
constexpr uint32_t kAccCol0 = 2 * kESlotCols;
constexpr int kTailBytes = 1024;
constexpr int kTQ = 16;                        // tile-queue slots (the producer runs < 8 tiles ahead)
constexpr int kMaxE = 20;                      // chunk partials per lane in the select (V <= 20 * 128 * 64)
constexpr int kTailDiv = 5;                    // the last fifth of a sweep's claims is kept in L2
constexpr size_t smem_bytes(int ring) {
  return 1024 + ring_nw(ring) * (size_t)kW2Stage + ring_nu(ring) * (size_t)kUStage +
         (size_t)kEpiWarps * kStagingPerWarp + kTailBytes;
}
static_assert(smem_bytes(kRingW2Deep) <= 232448 && smem_bytes(kRingUDeep) <= 232448, "shared memory per CTA");
// select scratch in the (idle) staging area: per team a row record, 16 words of
// exchange and four warps' 64 partial logits
constexpr int kSelRecOff = 0, kSelXwOff = 128, kSelRedOff = 256;
constexpr int kSelConfOff = kSelRedOff + 2 * kTeamWarps * 64 * 4;  // per team four warp sums of z
static_assert(kSelConfOff + 2 * kTeamWarps * 4 <= kEpiWarps * kStagingPerWarp, "select scratch");

struct Params {
  int B, G, V, r, H;
  int ntiles, nparts, ctas_per_m, n_ctas, n_mtiles;
  int ept;                   // chunk partials per select lane: E = ceil(nparts / 128)
  int pstride;               // row stride of part: 128 E
  uint64_t seed;
  const __nv_bfloat16* U;    // [B, G, V] (the select's chunk recompute)
  const __nv_bfloat16* W1;   // [V, r]
  const __nv_bfloat16* W2;   // [r, V]
  const __nv_bfloat16* w;    // [H + r]
  const __nv_bfloat16* h;    // [B, G, H] hidden states of the confidence head
  const int32_t* anchor;     // [B]
  const float* temp;         // [B]
  const uint32_t* req_id;    // [B]
  float2* rowstat;           // [B] (m, S) of the last selected position
  int32_t* tokens;           // [B, G]
  float2* part;              // [B, pstride] (max, sum) of a sampled row's chunk j, (value, index) of a
                             // greedy row's, at (j % E) 128 + j / E: the select's lanes read it coalesced
  float* pd_tok;
  float* pd_rows;            // [B, G, V]: stored directly by the small-batch form (TMA stores otherwise)
  int write_pd;              // 0: no p_d rows (no W items; p_d(x) and (m, S) come from the select)
  float2* pd_stat;           // [B, G] (m, S) of every drawn row, or null
  float* conf_logit;
  float* conf;
  unsigned* gbar;            // grid barrier counter, zero at launch
  unsigned* sched;           // [G + 1, n_mtiles] tile claims of each sweep, zero at launch
  // A scheduler launched behind this kernel (programmatic dependent launch)
  // overlaps its last sweep: every CTA adds 1 to sel_done (release) once its
  // selects of the last position are done, then lets the dependent grid
  // launch; CTA `donor` leaves its share of the last sweep to the others and
  // exits, so that the scheduler finds a free SM.  sel_done = null, donor = -1:
  // no scheduler behind.
  unsigned* sel_done;
  int donor;
  WsHeader* hdr;
  // RNN head (rnn_E non-null): E_k = tanh(W_o z_k), z_k = [s_k; W1[x_{k-1}]; h_k]
  const __nv_bfloat16* W_rnn;  // [3r, 2r + H]: gate, candidate and output rows
  const float* rnn_P;          // [B, G, 3r]: W_rnn[:, 2r:] . h_k of every position
  float* rnn_S;                // [2][B, r] fp32 state: s_k in buffer k & 1
  __nv_bfloat16* rnn_E;        // [2][B, r] rows E_k in buffer k & 1
  unsigned* rnn_done;          // [G, n_mtiles] recurrent units finished, zero at launch
};


__device__ __forceinline__ void epi_sync() {
  __syncwarp();
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_acquire_s32(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_s32(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A token not yet chosen in this launch: every CTA sets the tokens of the rows
// it selects to this before the first grid barrier; a select publishes the
// chosen token (after the row's (m, S)) with a release store.
constexpr int kTokPending = -1;

// Waits (bounded) for the token at t; kTokPending if the wait gave up.
__device__ int token_wait(const int* t, volatile int* abort_flag) {
  int v = ld_acquire_s32(t);
  if (v != kTokPending) return v;
  const uint64_t t0 = ptx::globaltimer_ns();
  while ((v = ld_acquire_s32(t)) == kTokPending) {
    if (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitLimitNs) return kTokPending;
    __nanosleep(32);
  }
  return v;
}

__device__ __forceinline__ void prefetch_row(const __nv_bfloat16* row, int r) {
  for (int o = 0; o < r * 2; o += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(row) + o));
}

// grid-wide barrier of the epilogue threads of every (resident) CTA
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* addr, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
  return old;
}

__device__ bool grid_barrier(const Params& p, unsigned target, volatile int* abort_flag, volatile int* s_ok,
                             int epi_tid) {
  epi_sync();
  if (epi_tid == 0) {
    int ok = *abort_flag ? 0 : 1;
    // release: the CTA's writes (ordered before by the named barrier) become
    // visible with the arrival; acquire: the other CTAs' writes are visible
    // after it
    if (ok && atom_add_acq_rel(p.gbar, 1u) + 1u < target) {
      const uint64_t t0 = ptx::globaltimer_ns();
      while (ld_acquire(p.gbar) < target) {
        if (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
          ok = 0;
          break;
        }
        __nanosleep(32);
      }
    }
    *s_ok = ok;
  }
  epi_sync();
  return *s_ok != 0;
}

// named barrier of one select team (four warps)
__device__ __forceinline__ void team_sync(int team) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(2 + team), "n"(kTeamWarps * 32) : "memory");
}

// Confidence of position k of row b, split over a team's four warps
// ([DSpark] 方法细节, 置信度头): z = w_h . h_k + w_e . W1[x] with x = x_{k-1}
// (the anchor for k = 0), c = sigmoid(z).  The team's lane tl takes the
// 8-element groups tl, tl + 128, .. of h_k and w_h (H % 8 == 0), warp 1's lane
// l also elements 8 l .. 8 l + 7 of W1[x] and w_e (r <= 256).  The first
// kConfPer groups of h_k (read once, from HBM) are loaded when the select of
// the row begins (conf_issue), with no address that waits on another load;
// after the crossing chunk's recompute each warp adds its share with w_h (read
// by every row: from L2) while the walk publishes the token (conf_partial), so
// that no load of the confidence waits on the select's critical path; for
// H > 4096 the rest of h_k is loaded there.  Nothing in the kernel reads the
// confidences.
constexpr int kConfPer = 4;
struct ConfLoads {
  uint4 h[kConfPer];
};

__device__ __forceinline__ void conf_issue(const Params& p, int b, int k, int tw, int lane, ConfLoads& L) {
  const int tl = tw * 32 + lane;
  const uint4* hq = reinterpret_cast<const uint4*>(p.h + ((size_t)b * p.G + k) * p.H);
  const int n8 = p.H / 8;
#pragma unroll
  for (int u = 0; u < kConfPer; ++u) {
    const int i = tl + u * kTeamWarps * 32;
    L.h[u] = i < n8 ? __ldcs(hq + i) : make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b, float acc) {
  const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 fa = __bfloat1622float2(a2[t]), fb = __bfloat1622float2(b2[t]);
    acc = fmaf(fa.x, fb.x, acc);
    acc = fmaf(fa.y, fb.y, acc);
  }
  return acc;
}

// This warp's share of z, summed over the warp (every lane holds it); team
// warp 1 also adds w_e . W1[x] (x = x_{k-1}; the row is in L2: the walk that
// chose x prefetched it).
__device__ __forceinline__ float conf_partial(const Params& p, int b, int k, int tw, int lane, const ConfLoads& L,
                                              int x) {
  const int tl = tw * 32 + lane;
  const int n8 = p.H / 8;
  float zh = 0.f;
  {
    // w_h is read by every row and position: it stays in L2
    const uint4* wq = reinterpret_cast<const uint4*>(p.w);
    uint4 wv[kConfPer];
#pragma unroll
    for (int u = 0; u < kConfPer; ++u) {
      const int i = tl + u * kTeamWarps * 32;
      wv[u] = i < n8 ? __ldg(wq + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kConfPer; ++u) zh = dot8_bf16(L.h[u], wv[u], zh);
  }
  if (n8 > kConfPer * kTeamWarps * 32) {
    const uint4* hq = reinterpret_cast<const uint4*>(p.h + ((size_t)b * p.G + k) * p.H);
    const uint4* wq = reinterpret_cast<const uint4*>(p.w);
    for (int i = tl + kConfPer * kTeamWarps * 32; i < n8; i += kTeamWarps * 32)
      zh = dot8_bf16(__ldcs(hq + i), __ldg(wq + i), zh);
  }
  if (tw == 1 && 8 * lane < p.r) {
    if (x < 0 || x >= p.V) x = 0;
    const uint4 e = *reinterpret_cast<const uint4*>(p.W1 + (size_t)x * p.r + 8 * lane);
    const uint4 we = __ldg(reinterpret_cast<const uint4*>(p.w + p.H + 8 * lane));
    zh = dot8_bf16(we, e, zh);
  }
  return warp_sum(zh);
}

// Row record of the select, in shared memory between its steps.
struct SelRec {
  int cstar;      // crossing chunk (sampled rows), -1 for greedy rows, -2 no row
  int hit;        // 1 if the running sum crossed u S
  float sbase;    // sum of 2^(y - m) over the chunks before cstar
  float target;   // u S
  float m, S;
  int b;
  int x;          // x_{k-1}, the token the logits condition on
  int tok;        // the chosen token
};

// The pass of the select of row b at position k over its chunk partials, by
// one team of four warps: lane tl = 32 tw + lane holds the partials
// [tl E, tl E + E) in token order.  Sampled rows: the row max m, the sum S of
// 2^(y - m), u = Philox(seed, req, k + 1, draw 0) and the 64-column chunk where
// the running sum in token order first exceeds u S ([DSpark] 方法细节, 草稿采样:
// inverse CDF), recorded for the recompute; (m, S) goes to rowstat.  Greedy
// rows get their token here (argmax, lowest id on ties), published with a
// release store.  The caller syncs the team before it reads the record.
__device__ void team_levels(const Params& p, int b, int k, int team, int tw, int lane, SelRec* rec, float* xw) {
  constexpr unsigned FULL = 0xffffffffu;
  const int E = p.ept;
  const int j0 = (tw * 32 + lane) * E;
  // partial j0 + t sits at t 128 + tl: each load is one coalesced row of the team
  const float2* P = p.part + (size_t)b * p.pstride + tw * 32 + lane;
  float2 e[kMaxE];
#pragma unroll
  for (int t = 0; t < kMaxE; ++t) {
    if (t >= E) break;  // uniform
    e[t] = (j0 + t < p.nparts) ? __ldcg(&P[t * 128]) : make_float2(-INFINITY, 0.f);
  }
  const float T = p.temp[b];
  const int xprev = (k == 0) ? p.anchor[b] : __ldcg(&p.tokens[(size_t)b * p.G + k - 1]);
  const uint32_t req = p.req_id[b];
  if (!(T > 0.f)) {
    float av = -INFINITY;
    int ai = INT_MAX;
#pragma unroll
    for (int t = 0; t < kMaxE; ++t) {
      if (t >= E) break;
      if (j0 + t < p.nparts) argmax_merge(av, ai, e[t].x, __float_as_int(e[t].y));
    }
    warp_argmax(av, ai);
    if (lane == 0) {
      xw[2 * tw] = av;
      xw[2 * tw + 1] = __int_as_float(ai);
    }
    team_sync(team);
    if (tw == 0 && lane == 0) {
      for (int w = 1; w < kTeamWarps; ++w) argmax_merge(av, ai, xw[2 * w], __float_as_int(xw[2 * w + 1]));
      p.rowstat[b] = make_float2(0.f, 1.f);
      if (p.pd_stat) p.pd_stat[(size_t)b * p.G + k] = make_float2(0.f, 1.f);
      if (!p.write_pd) p.pd_tok[(size_t)b * p.G + k] = 1.f;  // the one-hot row at the argmax
      if (ai >= 0 && ai < p.V) prefetch_row(p.W1 + (size_t)ai * p.r, p.r);  // for the E gathers
      st_release_s32(&p.tokens[(size_t)b * p.G + k], ai);
      rec->cstar = -1;
      rec->b = b;
      rec->x = xprev;
      rec->tok = ai;
    }
    return;
  }
  // the draw, while the partials are in flight
  const float u = philox_uniform(p.seed, req, (uint32_t)(k + 1), 0u);
  float ml = -INFINITY;
#pragma unroll
  for (int t = 0; t < kMaxE; ++t) {
    if (t >= E) break;
    ml = fmaxf(ml, e[t].x);
  }
  ml = warp_max(ml);
  if (lane == 0) xw[tw] = ml;
  team_sync(team);
  const float m = fmaxf(fmaxf(xw[0], xw[1]), fmaxf(xw[2], xw[3]));
  float sl = 0.f;
  int tlast = -1;
  float qm[kMaxE];  // each chunk's mass relative to m, reused by the walk below
#pragma unroll
  for (int t = 0; t < kMaxE; ++t) {
    if (t >= E) break;
    qm[t] = tile_mass(e[t].x, e[t].y, m);
    sl = __fadd_rn(sl, qm[t]);
    if (qm[t] > 0.f) tlast = t;
  }
  const float incl = warp_inclusive_scan(sl);
  const float up = __shfl_up_sync(FULL, incl, 1);
  const float excl = lane == 0 ? 0.f : up;
  const int jl = __reduce_max_sync(FULL, (unsigned)(tlast >= 0 ? j0 + tlast + 1 : 0));  // last positive + 1
  if (lane == 31) xw[4 + tw] = incl;
  if (lane == 0) xw[12 + tw] = __int_as_float(jl);
  team_sync(team);
  float wbase = 0.f, S = 0.f;
#pragma unroll
  for (int w = 0; w < kTeamWarps; ++w) {
    if (w == tw) wbase = S;
    S = __fadd_rn(S, xw[4 + w]);
  }
  int jlast = 0;
#pragma unroll
  for (int w = 0; w < kTeamWarps; ++w) jlast = max(jlast, __float_as_int(xw[12 + w]));
  jlast = max(jlast - 1, 0);
  const float target = u * S;
  const float ex = __fadd_rn(wbase, excl);
  const unsigned bal = __ballot_sync(FULL, j0 < p.nparts && __fadd_rn(wbase, incl) > target);
  if (lane == 0) xw[8 + tw] = __int_as_float(bal ? __ffs(bal) - 1 : 32);
  team_sync(team);
  int cw = -1, cl = 32;
#pragma unroll
  for (int w = kTeamWarps - 1; w >= 0; --w) {
    const int L = __float_as_int(xw[8 + w]);
    if (L < 32) {
      cw = w;
      cl = L;
    }
  }
  const bool writer = cw < 0 ? (tw == 0 && lane == 0) : (tw == cw && lane == cl);
  if (writer) {
    int cstar = -1;
    float cbase = 0.f;
    if (cw >= 0) {
      // the crossing lane walks its own chunks
      float run = ex;
#pragma unroll
      for (int t = 0; t < kMaxE; ++t) {
        if (t >= E) break;
        const float nr = __fadd_rn(run, tile_mass(e[t].x, e[t].y, m));
        if (cstar < 0 && j0 + t < p.nparts && nr > target) {
          cstar = j0 + t;
          cbase = run;
        }
        run = nr;
      }
    }
    const bool hit = cstar >= 0;
    // no crossing (reachable only through rounding): the last chunk with weight
    if (!hit) cstar = (cw >= 0 && tlast >= 0) ? j0 + tlast : jlast;
    // the walk reads the chunk's 64 U values of position k
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.U + ((size_t)b * p.G + k) * p.V + (size_t)cstar * CW));
    // (m, S) now: the walk's release of the token, after a team barrier, publishes it
    p.rowstat[b] = make_float2(m, S);
    if (p.pd_stat) p.pd_stat[(size_t)b * p.G + k] = make_float2(m, S);
    rec->cstar = cstar;
    rec->hit = hit ? 1 : 0;
    rec->sbase = cbase;
    rec->target = target;
    rec->m = m;
    rec->S = S;
    rec->b = b;
    rec->x = xprev;
  }
}

// The E_k . W2 part of the logits of chunk cstar of row b, split by rows of W2
// over a team of four warps: lane (j, c) of team warp tw takes columns
// 8 c .. 8 c + 7 of the rows tw r/4 + 4 i + j (128-bit loads, sixteen in flight),
// the four row phases j are added by shuffles, and red[tw][64] receives the
// warp's sums (fp32 fma in order within a phase).  erow: E_k of the row
// (W1[x_{k-1}] for the Markov head, the recurrent row for the RNN head).
__device__ void chunk_dot(const Params& p, const __nv_bfloat16* erow, int cstar, int tw, int lane, float* red) {
  constexpr unsigned FULL = 0xffffffffu;
  const int c8 = lane & 7, j = lane >> 3;
  const int v = cstar * CW + 8 * c8;
  const bool in = v < p.V;  // V % 8 == 0: the lane's eight columns are in or out together
  const int per = p.r / kTeamWarps;
  const int nt = per / 4;
  const int i0 = tw * per + j;
  const __nv_bfloat16* e = erow + i0;
  const __nv_bfloat16* w2 = p.W2 + (size_t)i0 * p.V + v;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int t0 = 0; t0 < nt; t0 += 16) {
    uint4 wv[16];
    float ev[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const bool ok = in && t0 + t < nt;
      wv[t] = ok ? __ldcg(reinterpret_cast<const uint4*>(w2 + (size_t)(4 * (t0 + t)) * p.V))
                 : make_uint4(0u, 0u, 0u, 0u);
      // (L2: the RNN head's rows are written during this launch)
      ev[t] = ok ? __bfloat162float(__ushort_as_bfloat16(__ldcg(reinterpret_cast<const unsigned short*>(e) +
                                                                4 * (t0 + t))))
                 : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const __nv_bfloat162* bp = reinterpret_cast<const __nv_bfloat162*>(&wv[t]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(bp[q]);
        a[2 * q] = fmaf(ev[t], f.x, a[2 * q]);
        a[2 * q + 1] = fmaf(ev[t], f.y, a[2 * q + 1]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    a[q] = __fadd_rn(a[q], __shfl_xor_sync(FULL, a[q], 8));
    a[q] = __fadd_rn(a[q], __shfl_xor_sync(FULL, a[q], 16));
  }
  if (j == 0) {
    float4* d = reinterpret_cast<float4*>(red + tw * 64 + 8 * c8);
    d[0] = make_float4(a[0], a[1], a[2], a[3]);
    d[1] = make_float4(a[4], a[5], a[6], a[7]);
  }
}

// The walk of the crossing chunk (one warp): l = U + sum of the warps' partial
// dot products, y = l c, w = 2^(y - m); the token is the first column whose
// running sum from sbase exceeds u S, else the chunk's last column with
// positive weight.  Writes the token and prefetches its W1 row.
__device__ void chunk_walk(const Params& p, const SelRec* rec, int k, int lane, const float* red, uint32_t upair) {
  constexpr unsigned FULL = 0xffffffffu;
  const int b = rec->b;
  const int v = rec->cstar * CW + 2 * lane;
  const bool in = v < p.V;
  const float c = row_scale(p.temp[b]);
  float w0 = 0.f, w1 = 0.f;
  if (in) {
    const __nv_bfloat162 uv = *reinterpret_cast<const __nv_bfloat162*>(&upair);
    float d0 = 0.f, d1 = 0.f;
    for (int w = 0; w < kTeamWarps; ++w) {
      d0 = __fadd_rn(d0, red[w * 64 + 2 * lane]);
      d1 = __fadd_rn(d1, red[w * 64 + 2 * lane + 1]);
    }
    const float2 fu = __bfloat1622float2(uv);
    w0 = exp_scaled(add_base(fu.x, d0), c, rec->m);
    w1 = exp_scaled(add_base(fu.y, d1), c, rec->m);
  }
  const float pair = __fadd_rn(w0, w1);
  const float incl = __fadd_rn(rec->sbase, warp_inclusive_scan(pair));
  const float up = __shfl_up_sync(FULL, incl, 1);
  const float ex = lane == 0 ? rec->sbase : up;
  int tok = -1;
  float wsel = 0.f;  // the chosen token's weight 2^(y - m)
  const unsigned over = __ballot_sync(FULL, rec->hit && incl > rec->target);
  if (over) {
    const int L = __ffs(over) - 1;
    if (lane == L) {
      tok = (__fadd_rn(ex, w0) > rec->target) ? v : v + 1;
      wsel = tok == v ? w0 : w1;
    }
    tok = __shfl_sync(FULL, tok, L);
    wsel = __shfl_sync(FULL, wsel, L);
  } else {
    const unsigned pos = __ballot_sync(FULL, w0 > 0.f || w1 > 0.f);
    if (pos) {
      const int L = 31 - __clz(pos);
      if (lane == L) {
        tok = (w1 > 0.f) ? v + 1 : v;
        wsel = (w1 > 0.f) ? w1 : w0;
      }
      tok = __shfl_sync(FULL, tok, L);
      wsel = __shfl_sync(FULL, wsel, L);
    } else {
      tok = rec->cstar * CW;  // no positive weight at all (unreachable for a crossing chunk)
    }
  }
  if (lane == 0) {
    // without p_d rows, p_d(x_k) comes from this walk (the W item writes it otherwise)
    if (!p.write_pd) p.pd_tok[(size_t)b * p.G + k] = __fmul_rn(wsel, inv_sum(rec->S));
    prefetch_row(p.W1 + (size_t)tok * p.r, p.r);  // for the E gathers
    st_release_s32(&p.tokens[(size_t)b * p.G + k], tok);
    const_cast<SelRec*>(rec)->tok = tok;
  }
}

// RNN head: the recurrent step of position k for the units this CTA owns
// ([DSpark] 方法细节, "RNN头的实现").  A unit is 32 rows x C state columns
// (C = 4 in the 128-row form, 2 in the small-batch form, whose shared memory
// is smaller); units are numbered column groups fastest, and CTA c owns the
// contiguous range [c n / n_ctas, (c + 1) n / n_ctas), so that consecutive
// units of a CTA mostly share their rows and z' stays in registers.  The
// unit's 3 C weight rows are staged in scr as fp32, [2r][3C] per z' entry
// (gate g, column c at C g + c), each 64-entry segment offset by 16 bytes so
// that the eight segments' reads fall in distinct banks.  Eight epilogue
// threads per row: thread s sums z' entries 64 s .. 64 s + 63 of
// z' = [s_k; W1[x_{k-1}]] (fp32 fma chains in ascending order), the eight sums
// are added by a fixed shuffle tree (the lower lane's first), then thread
// c < C finishes column c:
//     pre = W_rnn[:, :2r] z' + P[b, k],  g = sigmoid(pre_g),
//     s_{k+1} = g s_k + (1 - g) tanh(pre_c),  E_k = tanh(pre_o) (bf16),
// s_0 = 0 and x_{-1} the anchor.  After its last unit the CTA adds, with
// release semantics, its unit count of each M-tile m to rnn_done[k, m].
// False if a token wait gave up.
constexpr int kRnnRows = 32;
template <int C>
struct RnnUnit {
  static constexpr int kSegBytes = 64 * 3 * C * 4 + 16;  // one segment of staged weights (fp32), padded
  static constexpr int kStageLd = (3 * C * 512 / 8 + kEpiThreads - 1) / kEpiThreads;  // 16-byte loads per thread
  static constexpr int kScrBytes = 8 * kSegBytes + kRnnRows * 64;  // segments, then a float4 x 4 slot per row
};
constexpr int kWideRnnCols = 4;  // state columns of a unit in the 128-row form
static_assert(RnnUnit<kWideRnnCols>::kScrBytes <= kEpiWarps * kStagingPerWarp, "unit scratch in the p_d staging");

template <int kRnnCols>
__device__ bool rnn_units(const Params& p, int k, uint8_t* scr, int epi_tid, volatile int* abort_flag) {
  constexpr int kRnnSegBytes = RnnUnit<kRnnCols>::kSegBytes;
  constexpr int kRnnStageLd = RnnUnit<kRnnCols>::kStageLd;
  constexpr unsigned FULL = 0xffffffffu;
  const int r = p.r, K = 2 * r, ldw = 2 * r + p.H, B = p.B;
  const int nrb = (B + kRnnRows - 1) / kRnnRows;  // row blocks
  const int ncg = r / kRnnCols;
  const int nunits = nrb * ncg;
  const int u_lo = (int)((long long)nunits * blockIdx.x / p.n_ctas);
  const int u_hi = (int)((long long)nunits * (blockIdx.x + 1) / p.n_ctas);
  const int seg = epi_tid & 7;   // this thread's 64-entry segment of z'
  const int rr = epi_tid >> 3;   // this thread's row of the unit
  const int i0 = seg * 64;
  const int nld = 3 * kRnnCols * (K / 8);  // 16-byte pieces of a unit's weight rows
  bool ok = true;
  // the weight rows of column group cg, piece idx = epi_tid + kEpiThreads j:
  // row (gate g, column cc) = idx % 12, eight entries from 8 (idx / 12)
  uint4 wq[kRnnStageLd];
  auto load_w = [&](int cg) {
#pragma unroll
    for (int j = 0; j < kRnnStageLd; ++j) {
      const int idx = epi_tid + j * kEpiThreads;
      if (idx < nld) {
        const int rowi = idx % (3 * kRnnCols), s8 = idx / (3 * kRnnCols);
        const int g = rowi / kRnnCols, cc = rowi - g * kRnnCols;
        wq[j] = __ldg(reinterpret_cast<const uint4*>(p.W_rnn + (size_t)(g * r + cg * kRnnCols + cc) * ldw) + s8);
      }
    }
  };
  for (int u = u_lo; u < u_hi;) {
    // the units of one row block share z' = [s_k; W1[x_{k-1}]] of its rows
    const int rb = u / ncg;
    const int u_end = min(u_hi, (rb + 1) * ncg);
    const int b = rb * kRnnRows + rr;
    const bool used = b < B && i0 < K;  // a segment past 2r (r < 256) loads and adds nothing
    float z[64];
    if (used && i0 < r) {
      if (k > 0) {
        const float4* sq = reinterpret_cast<const float4*>(p.rnn_S + ((size_t)(k & 1) * B + b) * r + i0);
        float4 v[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = __ldcg(sq + q);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          z[4 * q] = v[q].x;
          z[4 * q + 1] = v[q].y;
          z[4 * q + 2] = v[q].z;
          z[4 * q + 3] = v[q].w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 64; ++q) z[q] = 0.f;  // s_0 = 0
      }
    } else if (used) {
      int x = (k == 0) ? p.anchor[b] : token_wait(&p.tokens[(size_t)b * p.G + k - 1], abort_flag);
      if (x == kTokPending) {
        ok = false;
        x = 0;
      }
      if (x < 0 || x >= p.V) x = 0;  // reported by the gather
      const uint4* wp = reinterpret_cast<const uint4*>(p.W1 + (size_t)x * r + (i0 - r));
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = __ldg(wp + q);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v[q]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h2[e]);
          z[8 * q + 2 * e] = f.x;
          z[8 * q + 2 * e + 1] = f.y;
        }
      }
    } else {
#pragma unroll
      for (int q = 0; q < 64; ++q) z[q] = 0.f;
    }
  for (; u < u_end; ++u) {
    const int cg = u - rb * ncg;
    const int col0 = cg * kRnnCols;
    load_w(cg);
    // the finishing operands of the row's kRnnCols columns, copied by its
    // segment-0 thread into the row's slot: the aligned four columns that
    // hold them, of P[b, k] per gate, then of s_k
    float4* fslot = reinterpret_cast<float4*>(scr + 8 * kRnnSegBytes) + 4 * rr;
    const int c4 = col0 & ~3;
    if (seg == 0 && b < B) {
      if (p.rnn_P) {
        const float* pr = p.rnn_P + ((size_t)b * p.G + k) * 3 * r + c4;
        ptx::cp_async16_cg(fslot, pr);
        ptx::cp_async16_cg(fslot + 1, pr + r);
        ptx::cp_async16_cg(fslot + 2, pr + 2 * r);
      } else {
        fslot[0] = fslot[1] = fslot[2] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (k > 0)
        ptx::cp_async16_cg(fslot + 3, p.rnn_S + ((size_t)(k & 1) * B + b) * r + c4);
      else
        fslot[3] = make_float4(0.f, 0.f, 0.f, 0.f);  // s_0 = 0
    }
    // stage this unit's weight rows: entry (i, rowi) at segment i / 64, slot (i % 64) 12 + rowi
#pragma unroll
    for (int j = 0; j < kRnnStageLd; ++j) {
      const int idx = epi_tid + j * kEpiThreads;
      if (idx < nld) {
        const int rowi = idx % (3 * kRnnCols), s8 = idx / (3 * kRnnCols);
        const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&wq[j]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int i = s8 * 8 + e;
          reinterpret_cast<float*>(scr + (i >> 6) * kRnnSegBytes)[(i & 63) * 3 * kRnnCols + rowi] =
              __bfloat162float(hv[e]);
        }
      }
    }
    epi_sync();
    float acc[3 * kRnnCols];
#pragma unroll
    for (int a = 0; a < 3 * kRnnCols; ++a) acc[a] = 0.f;
    if (used) {
      const uint8_t* wseg = scr + seg * kRnnSegBytes;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        if constexpr (kRnnCols == 4) {
          const float4* w = reinterpret_cast<const float4*>(wseg + i * 3 * kRnnCols * 4);
#pragma unroll
          for (int h = 0; h < 3; ++h) {
            const float4 f = w[h];
            acc[4 * h] = fmaf(f.x, z[i], acc[4 * h]);
            acc[4 * h + 1] = fmaf(f.y, z[i], acc[4 * h + 1]);
            acc[4 * h + 2] = fmaf(f.z, z[i], acc[4 * h + 2]);
            acc[4 * h + 3] = fmaf(f.w, z[i], acc[4 * h + 3]);
          }
        } else {
          const float2* w = reinterpret_cast<const float2*>(wseg + i * 3 * kRnnCols * 4);
#pragma unroll
          for (int h = 0; h < 3 * kRnnCols / 2; ++h) {
            const float2 f = w[h];
            acc[2 * h] = fmaf(f.x, z[i], acc[2 * h]);
            acc[2 * h + 1] = fmaf(f.y, z[i], acc[2 * h + 1]);
          }
        }
      }
    }
    // the eight segments' sums, lower lane first at every level
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
      for (int a = 0; a < 3 * kRnnCols; ++a) {
        const float v = __shfl_xor_sync(FULL, acc[a], o);
        acc[a] = (seg & o) ? __fadd_rn(v, acc[a]) : __fadd_rn(acc[a], v);
      }
    if (seg == 0 && b < B) ptx::cp_async_wait_all();
    __syncwarp();  // the slot's copies seen by the row's other threads
    if (b < B && seg < kRnnCols) {
      const float* fs = reinterpret_cast<const float*>(fslot) + (col0 - c4);
      float pg = fs[seg], pc = fs[4 + seg], po = fs[8 + seg];
      const float sp = fs[12 + seg];
#pragma unroll
      for (int c = 0; c < kRnnCols; ++c)
        if (c == seg) {
          pg += acc[c];
          pc += acc[kRnnCols + c];
          po += acc[2 * kRnnCols + c];
        }
      const int col = col0 + seg;
      const float gt = 1.f / (1.f + expf(-pg));
      p.rnn_S[((size_t)((k + 1) & 1) * B + b) * r + col] = gt * sp + (1.f - gt) * tanhf(pc);
      p.rnn_E[((size_t)(k & 1) * B + b) * r + col] = __float2bfloat16_rn(tanhf(po));
    }
    // every read of scr before the next unit's staging
    epi_sync();
  }
  }
  // every write of the units before the counts (the last epi_sync above
  // orders them before thread 0's release)
  if (epi_tid == 0 && u_lo < u_hi) {
    constexpr int kRbPerTile = BM / kRnnRows;
    const int m_lo = (u_lo / ncg) / kRbPerTile, m_hi = ((u_hi - 1) / ncg) / kRbPerTile;
    for (int m = m_lo; m <= m_hi; ++m) {
      const int a0 = max(u_lo, m * kRbPerTile * ncg), a1 = min(u_hi, (m + 1) * kRbPerTile * ncg);
      atom_add_acq_rel(&p.rnn_done[(size_t)k * p.n_mtiles + m], (unsigned)(a1 - a0));
    }
  }
  return ok;
}

// The select of position k for the rows this CTA serves (rows blockIdx.x +
// n_ctas j), by the epilogue's two teams of four warps (team t takes j = t,
// t + 2, ..): the pass over the row's chunk partials, then for a sampled row
// the recompute of the crossing chunk and its walk, and the confidence of the
// position.  scr: the teams' scratch in shared memory.
__device__ __forceinline__ void select_rows(const Params& p, int k, uint8_t* scr, int team, int tw, int lane) {
  const int G = p.G;
  SelRec* rec = reinterpret_cast<SelRec*>(scr + kSelRecOff) + team;
  float* xw = reinterpret_cast<float*>(scr + kSelXwOff) + team * 16;
  float* red = reinterpret_cast<float*>(scr + kSelRedOff) + team * kTeamWarps * 64;
  float* cz = reinterpret_cast<float*>(scr + kSelConfOff) + team * kTeamWarps;
  for (int j = team;; j += 2) {
    const int rb = (int)blockIdx.x + p.n_ctas * j;
    if (rb >= p.B) break;
    // the confidence of (rb, k) needs x_{k-1} only: its loads go out first
    // and land during the levels pass
    ConfLoads cl;
    conf_issue(p, rb, k, tw, lane, cl);
    team_levels(p, rb, k, team, tw, lane, rec, xw);
    team_sync(team);
    const int cstar = rec->cstar;
    uint32_t upair = 0u;
    if (cstar >= 0) {
      // the walking warp fetches the chunk's U pairs (prefetched to L2 by the
      // levels pass) with the recompute's loads
      if (tw == 0 && cstar * CW + 2 * lane < p.V)
        upair = __ldcg(reinterpret_cast<const unsigned*>(p.U + ((size_t)rb * G + k) * p.V + cstar * CW + 2 * lane));
      // E_k of the row: the recurrent row (RNN head) or W1[x_{k-1}]
      const int xk = (rec->x < 0 || rec->x >= p.V) ? 0 : rec->x;
      const __nv_bfloat16* erow = p.rnn_E ? p.rnn_E + ((size_t)(k & 1) * p.B + rb) * p.r : p.W1 + (size_t)xk * p.r;
      chunk_dot(p, erow, cstar, tw, lane, red);
      team_sync(team);
      if (tw == 0) chunk_walk(p, rec, k, lane, red, upair);
    }
    // this warp's share of the confidence, off the walk's path: warps 1-3
    // while warp 0 walks, warp 0 after it (the loads have landed by now)
    {
      const float zp = conf_partial(p, rb, k, tw, lane, cl, rec->x);
      if (lane == 0) cz[tw] = zp;
    }
    // the record, exchange words and partial logits are free for the next row
    team_sync(team);
    if (tw == 1 && lane == 0) {
      const float z = (cz[0] + cz[1]) + (cz[2] + cz[3]);
      p.conf_logit[(size_t)rb * G + k] = z;
      p.conf[(size_t)rb * G + k] = 1.f / (1.f + expf(-z));
    }
  }
  // every warp is done with the scratch before it is reused
  epi_sync();
}

// kRnn: the RNN head's rows (recurrent units in each gather); else W1 rows.
// kRing: the stage rings (kRingW2Deep or kRingUDeep).
template <bool kRnn, int kRing>
__global__ void __launch_bounds__(kThreads, 1)
    k_draft_fused(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmW2,
                  const __grid_constant__ CUtensorMap tmPd, Params p) {
  constexpr int NW = ring_nw(kRing), NU = ring_nu(kRing);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int r = p.r;
  const int nkc = r / KC;
  uint8_t* sW = smem;
  uint8_t* sU = sW + NW * kW2Stage;
  uint8_t* sStg = sU + NU * kUStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + kEpiWarps * kStagingPerWarp);
  uint64_t* fullW = bars;
  uint64_t* emptyW = fullW + NW;
  uint64_t* fullU = emptyW + NW;
  uint64_t* emptyU = fullU + NU;
  uint64_t* tfull = emptyU + NU;
  uint64_t* tempty = tfull + 2;
  uint64_t* eready = tempty + 2;
  uint64_t* mma_done = eready + 1;
  uint64_t* tqfull = mma_done + 1;  // [kTQ]
  volatile int* tq = reinterpret_cast<volatile int*>(tqfull + kTQ);  // [kTQ] tile of each queue entry, -1 ends a sweep
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tq) + kTQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = abort_flag + 1;
  volatile int* e_seen = s_ok + 1;  // gathers the MMA issuer has waited for

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = (int)blockIdx.x / p.ctas_per_m;
  const int row_base = m_tile * BM;
  const int G = p.G;
  // sweep q = 0 .. G: q = 0 is S(0) alone; q >= 1 is W(q - 1) + S(q) (no S in
  // the last).  The CTAs of an M-tile claim its vocabulary tiles one at a time
  // from a counter per sweep (the producer claims, and hands each tile to the
  // MMA issuer and the epilogue through the tile queue); sweeps alternate the
  // claim order, so that each starts on the tiles the previous one read last.
  auto tile_of = [&](unsigned i, int q) {
    return i >= (unsigned)p.ntiles ? -1 : ((q & 1) ? p.ntiles - 1 - (int)i : (int)i);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NW; ++s) {
      ptx::mbar_init(&fullW[s], 1);
      ptx::mbar_init(&emptyW[s], 1);
    }
    for (int s = 0; s < NU; ++s) {
      ptx::mbar_init(&fullU[s], 1);
      ptx::mbar_init(&emptyU[s], kEpiWarps);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], kEpiWarps);
    }
    ptx::mbar_init(eready, kEpiWarps);
    ptx::mbar_init(mma_done, 1);
    for (int j = 0; j < kTQ; ++j) ptx::mbar_init(&tqfull[j], 1);
    *abort_flag = 0;
    *e_seen = 0;
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
      // L2 policies: a sweep's last kTailDiv-th of claims are the next sweep's
      // first (the claim order alternates), so their W2 tile and the U rows of
      // their S item (read again by the next sweep's W item) are kept
      // (evict-last); other U rows are read for the last time (evict-first);
      // other W2 tiles need to last only until the other M-tile's CTA has read
      // them (evict-normal)
      const uint64_t pol_last = ptx::policy_evict_last();
      const uint64_t pol_first = ptx::policy_evict_first();
      const uint64_t pol_normal = ptx::policy_evict_normal();
      const unsigned tail0 = (unsigned)(p.ntiles - p.ntiles / kTailDiv);
      int iw = 0, iu = 0, jq = 0;
      bool ok = true;
      for (int q = 0; q < G + p.write_pd && ok; ++q) {
        const int s = q - 1;
        const bool hasW = p.write_pd && s >= 0, hasS = s + 1 < G;
        unsigned* claim = p.sched + (size_t)q * p.n_mtiles + m_tile;
        // the donor CTA claims nothing in the last sweep (q = G has W items only)
        const bool donate = q == G && (int)blockIdx.x == p.donor;
        unsigned ci = donate ? (unsigned)p.ntiles : atomicAdd(claim, 1u);  // claim index of the tile n
        int n = tile_of(ci, q);
        while (ok) {
          // hand the tile (or the end of the sweep) to the MMA issuer and the
          // epilogue; the arrive releases the queue entry
          tq[jq % kTQ] = n;
          ptx::mbar_arrive(&tqfull[jq % kTQ]);
          ++jq;
          if (n < 0) break;
          const int v0 = n * BN;
          const bool keep = ci >= tail0;
          ci = atomicAdd(claim, 1u);  // the next claim, in flight during the loads
          n = tile_of(ci, q);
          for (int kc = 0; kc < nkc; ++kc, ++iw) {
            const int st = iw % NW;
            if (!ptx::mbar_wait(&emptyW[st], ((iw / NW) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            uint8_t* dst = sW + st * kW2Stage;
            ptx::mbar_expect_tx(&fullW[st], kW2Stage);
            for (int c = 0; c < NCH; ++c)
              ptx::tma_load_2d(dst + c * (KC * CW * 2), &tmW2, &fullW[st], v0 + c * CW, kc * KC,
                               keep ? pol_last : pol_normal);
          }
          for (int item = 0; item < 2 && ok; ++item) {
            if (item == 0 ? !hasW : !hasS) continue;
            const int kk = item == 0 ? s : s + 1;
            const int su = iu % NU;
            if (!ptx::mbar_wait(&emptyU[su], ((iu / NU) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            ptx::mbar_expect_tx(&fullU[su], kUStage);
            for (int c = 0; c < NCH; ++c)
              ptx::tma_load_3d(sU + su * kUStage + c * kUChunk, &tmU, &fullU[su], v0 + c * CW, kk, row_base,
                               (keep && item == 1) ? pol_last : pol_first);
            ++iu;
          }
        }
      }
      if (!ok) fail();
      for (int j = max(0, iw - NW); j < iw; ++j) ptx::mbar_wait(&fullW[j % NW], (j / NW) & 1, abort_flag, kWaitLimitNs);
      for (int j = max(0, iu - NU); j < iu; ++j) ptx::mbar_wait(&fullU[j % NU], (j / NU) & 1, abort_flag, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, false, true);
      int it = 0, iw = 0, jq = 0;
      bool ok = true;
      // E_q of sweep q's S items: the q-th gather.  Waited for in every such
      // sweep, with tiles or without, so that no phase of eready is skipped.
      auto wait_e = [&](int q) {
        if (!ptx::mbar_wait(eready, (uint32_t)(q & 1), abort_flag, kWaitLimitNs)) return false;
        *e_seen = q + 1;
        return true;
      };
      for (int q = 0; q < G + p.write_pd && ok; ++q) {
        const int s = q - 1;
        const bool hasW = p.write_pd && s >= 0, hasS = s + 1 < G;
        bool e_ok = false;
        while (ok) {
          if (!ptx::mbar_wait(&tqfull[jq % kTQ], (jq / kTQ) & 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const int n = tq[jq % kTQ];
          ++jq;
          if (n < 0) {
            if (hasS && !e_ok) ok = wait_e(q);
            break;
          }
          bool staged = false;  // this tile's W2 stages waited for
          for (int item = 0; item < 2 && ok; ++item) {
            if (item == 0 ? !hasW : !hasS) continue;
            if (item == 1 && !e_ok) {
              if (!wait_e(q)) {
                ok = false;
                break;
              }
              e_ok = true;
            }
            const int a = it & 1;
            if (!ptx::mbar_wait(&tempty[a], ((it >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const int kk = item == 0 ? s : s + 1;
            const uint32_t a_base = tmem + (uint32_t)((kk & 1) * kESlotCols);
            const uint32_t d = tmem + kAccCol0 + (uint32_t)(a * BN);
            for (int kc = 0; kc < nkc; ++kc) {
              const int st = (iw + kc) % NW;
              if (!staged) {
                if (!ptx::mbar_wait(&fullW[st], ((iw + kc) / NW) & 1, abort_flag, kWaitLimitNs)) {
                  ok = false;
                  break;
                }
                ptx::tc_fence_after();
              }
              const uint32_t aW2 = ptx::smem_u32(sW + st * kW2Stage);
#pragma unroll
              for (int k4 = 0; k4 < KC / 16; ++k4) {
                const int ks = kc * (KC / 16) + k4;
                // B: W2 K-chunk [64 x 128], MN-major, 128B swizzle: two 64-column
                //    blocks 8 KB apart; 8-row groups 1024 B apart along K
                const uint64_t bd = ptx::smem_desc_sw128(aW2 + k4 * 2048, KC * CW * 2, 1024);
                ptx::tc_mma_tmem_a(d, a_base + (uint32_t)(ks * 8), bd, idesc, ks > 0 ? 1u : 0u);
              }
            }
            if (!ok) break;
            staged = true;
            ptx::tc_commit(&tfull[a]);
            ++it;
          }
          if (!ok) break;
          // the tile's W2 stages are free once both of its products are done
          for (int kc = 0; kc < nkc; ++kc) ptx::tc_commit(&emptyW[(iw + kc) % NW]);
          iw += nkc;
        }
      }
      if (!ok) fail();
      ptx::tc_commit(mma_done);
      ptx::mbar_wait(mma_done, 0, abort_flag, kWaitLimitNs);
    }
  } else {
    // ------------------------------ epilogue ----------------------------------
    const int ew = warp - kEpiWarp0;
    const int epi_tid = ew * 32 + lane;
    const int g = ew >> 2;
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const int b = row_base + row;
    const bool vrow = b < p.B;
    const bool wlive = row_base + qd * 32 < p.B;  // warp-uniform: some row of this warp is in the batch
    const uint32_t lane_bits = (uint32_t)(qd * 32) << 16;
    const int npieces = r / 64;
    const float T_ = vrow ? p.temp[b] : 1.f;
    const bool sampled = T_ > 0.f;
    const float c = row_scale(T_);
    uint8_t* stg = sStg + ew * kStagingPerWarp;
    const uint64_t pol_keep = ptx::policy_evict_last();
    unsigned nbar = 0;
    int it = 0, iu = 0, jq = 0;
    bool alive = true;

    // E_k = W1[x_{k-1}] (x_0 = anchor) into TMEM slot k & 1
    // the next W item's row data, taken by the gather that waits for its token:
    // x_{k-1} and (m, S) of position k - 1 (published before the token)
    int wx = -1;
    float2 wst = make_float2(0.f, 1.f);
    auto gather = [&](int k) {
      int x = 0;
      if (vrow) {
        if (k == 0) {
          x = p.anchor[b];
        } else {
          x = token_wait(&p.tokens[(size_t)b * p.G + k - 1], abort_flag);
          if (x == kTokPending) {
            fail();
            x = 0;
          }
          wx = x;
          wst = __ldcg(&p.rowstat[b]);
        }
        if (x < 0 || x >= p.V) {
          if (g == 0) report_error(p.hdr, DSPARK_BAD_INPUT, x);
          x = 0;
        }
      }
      const uint4* src = reinterpret_cast<const uint4*>(p.W1 + (size_t)x * r);
      if constexpr (kRnn) {
        // the recurrent units of position k, then this M-tile's rows E_k once
        // every unit of the M-tile has finished
        if (!rnn_units<kWideRnnCols>(p, k, sStg, epi_tid, abort_flag)) fail();
        if (epi_tid == 0) {
          // the units of this M-tile: its row blocks x the column groups
          const int rb_hi = min((m_tile + 1) * BM, ((p.B + kRnnRows - 1) / kRnnRows) * kRnnRows);
          const unsigned target = (unsigned)((rb_hi - m_tile * BM) / kRnnRows * (r / kWideRnnCols));
          const unsigned* cnt = p.rnn_done + (size_t)k * p.n_mtiles + m_tile;
          int okw = *abort_flag ? 0 : 1;
          const uint64_t t0 = ptx::globaltimer_ns();
          while (okw && ld_acquire(cnt) < target) {
            if (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitLimitNs) okw = 0;
            __nanosleep(32);
          }
          *s_ok = okw;
        }
        epi_sync();
        if (!*s_ok && epi_tid == 0) fail();
        src = reinterpret_cast<const uint4*>(p.rnn_E + ((size_t)(k & 1) * p.B + (vrow ? b : 0)) * r);
      }
      const uint32_t slot = tmem + lane_bits + (uint32_t)((k & 1) * kESlotCols);
      // group g copies the 64-element pieces g, g + 2 of its rows (all loads
      // in flight before the first store)
      constexpr int kPer = 2 * kESlotCols / 64 / kGroups;
      uint32_t wv[kPer][32];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int pc = g + i * kGroups;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          // (L2 for the RNN head's rows: written during this launch)
          const uint4 qv = (vrow && pc < npieces) ? (kRnn ? __ldcg(src + pc * 8 + e) : src[pc * 8 + e])
                                                  : make_uint4(0u, 0u, 0u, 0u);
          wv[i][4 * e] = qv.x;
          wv[i][4 * e + 1] = qv.y;
          wv[i][4 * e + 2] = qv.z;
          wv[i][4 * e + 3] = qv.w;
        }
      }
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int pc = g + i * kGroups;
        if (pc < npieces) {  // warp-uniform
          __syncwarp();
          ptx::tmem_st32(slot + (uint32_t)(pc * 32), wv[i]);
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // the MMA issuer has waited for the previous gather, so that no phase
        // of eready runs ahead of it (a CTA may get no tile in a sweep)
        const uint64_t t0 = ptx::globaltimer_ns();
        while (*e_seen < k) {
          if (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            fail();
            break;
          }
          __nanosleep(32);
        }
        ptx::mbar_arrive(eready);
      }
    };

    const int team = ew / kTeamWarps, tw = ew % kTeamWarps;
    auto select = [&](int k) { select_rows(p, k, sStg, team, tw, lane); };

    // tokens of the rows this CTA selects: not chosen yet (ordered before
    // every wait on them by the first grid barrier)
    for (int rb = (int)blockIdx.x + p.n_ctas * ew; rb < p.B; rb += p.n_ctas * kEpiWarps)
      for (int k = lane; k < G; k += 32) p.tokens[(size_t)rb * G + k] = kTokPending;
    if (!*abort_flag) gather(0);
    for (int q = 0; q < G + p.write_pd && alive; ++q) {
      const int s = q - 1;
      const bool hasW = p.write_pd && s >= 0, hasS = s + 1 < G;
      // W(s) row data: (m, 1/S) and the token x_s (chosen by the select)
      float rm = 0.f, rinvS = 1.f;
      int xs = -1;
      if (hasW && vrow) {
        // the select of another CTA published (m, S) and then x_s; the gather of
        // E_{s+1} waited for x_s and read both
        xs = wx;
        rm = wst.x;
        rinvS = inv_sum(wst.y);
      }
      float pdtok = 0.f;
      bool have_pdtok = false;
      const int ch = g;
      bool tiles_ok = true;
      while (tiles_ok) {
        // the next tile this CTA claimed, or the end of the sweep
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&tqfull[jq % kTQ], (jq / kTQ) & 1, abort_flag, kWaitLimitNs))) {
          if (lane == 0) fail();
          tiles_ok = false;
          break;
        }
        const int n = tq[jq % kTQ];
        ++jq;
        if (n < 0) break;
        const int v0 = n * BN + ch * CW;
        const int nvalid = min(CW, p.V - v0);
        for (int item = 0; item < 2; ++item) {
          if (item == 0 ? !hasW : !hasS) continue;
          const int a = it & 1;
          bool ok = ptx::mbar_wait(&tfull[a], (it >> 1) & 1, abort_flag, kWaitLimitNs);
          const int su = iu % NU;
          if (ok) ok = ptx::mbar_wait(&fullU[su], (iu / NU) & 1, abort_flag, kWaitLimitNs);
          if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) fail();
            tiles_ok = false;
            break;
          }
          ++it;
          ++iu;
          ptx::tc_fence_after();
          if (!wlive) {
            // every row of this warp is past the batch: release the accumulator
            // and the U stage unread
            __syncwarp();
            if (lane == 0) {
              ptx::mbar_arrive(&tempty[a]);
              ptx::mbar_arrive(&emptyU[su]);
            }
            continue;
          }
          const uint32_t ta = tmem + lane_bits + kAccCol0 + (uint32_t)(a * BN + ch * CW);
          const uint8_t* su_row = sU + su * kUStage + ch * kUChunk + row * 128;
          // the row's 64 U values (8 x 16 B, 128-byte swizzle), loaded before the
          // TMEM wait so that the two latencies overlap
          uint4 uq[8];
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) uq[c8] = *reinterpret_cast<const uint4*>(su_row + ((c8 ^ (row & 7)) << 4));
          // logits of the chunk's 64 columns: accumulator + U; reading the
          // accumulator releases it
          float x[64];
          {
            float (&xa)[32] = *reinterpret_cast<float(*)[32]>(&x[0]);
            float (&xb)[32] = *reinterpret_cast<float(*)[32]>(&x[32]);
            __syncwarp();
            ptx::tmem_ld32(ta, xa);
            ptx::tmem_ld32(ta + 32, xb);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[a]);
          }
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const __nv_bfloat162* bp = reinterpret_cast<const __nv_bfloat162*>(&uq[c8]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(bp[e]);
              x[8 * c8 + 2 * e] = add_base(f.x, x[8 * c8 + 2 * e]);
              x[8 * c8 + 2 * e + 1] = add_base(f.y, x[8 * c8 + 2 * e + 1]);
            }
          }
          if (item == 1) {
            // the U stage's next fill is an async-proxy (TMA) write: order this
            // warp's generic reads of it before the release
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&emptyU[su]);
            // S item: chunk partial of position s + 1
            float2 part;
            if (sampled) {
              // chunk max on the logits (l c is monotone in l for c > 0), then
              // the sum of 2^(l c - m_chunk); columns past V count as -inf
              if (nvalid < CW) {
#pragma unroll
                for (int j = 0; j < CW; ++j)
                  if (j >= nvalid) x[j] = -INFINITY;
              }
              float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
              for (int j = 0; j < CW; ++j) mx[j & 3] = fmaxf(mx[j & 3], x[j]);
              const float lm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
              float cs = 0.f, mh = -INFINITY;
              if (lm != -INFINITY) {
                mh = scale_logit(lm, c);
                float sm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < CW; ++j) sm[j & 3] += exp_scaled(x[j], c, mh);
                cs = (sm[0] + sm[1]) + (sm[2] + sm[3]);
              }
              part = make_float2(mh, cs);
            } else {
              float av = -INFINITY;
              int ai = INT_MAX;
#pragma unroll
              for (int j = 0; j < CW; ++j)
                if (j < nvalid && x[j] > av) {
                  av = x[j];
                  ai = v0 + j;
                }
              part = make_float2(av, __int_as_float(ai));
            }
            // the select reads the partials right after the sweep: keep them in L2
            // (evict-last) through the sweep's streams (evict-first)
            if (v0 < p.V && vrow)
              ptx::st_global_hint(&p.part[(size_t)b * p.pstride + (v0 / CW) % p.ept * 128 + (v0 / CW) / p.ept], part,
                                  pol_keep);
          } else {
            // W item: p_d^s = 2^(l c - m) / S (one-hot for greedy rows); columns
            // past V are computed but not stored (the TMA store clips them)
            const int row0 = row_base + qd * 32;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float* xh = x + 32 * h;
              if (sampled) {
#pragma unroll
                for (int j = 0; j < 32; ++j) xh[j] = __fmul_rn(exp_scaled(xh[j], c, rm), rinvS);
              }
              const int jx = xs - (v0 + 32 * h);
              if (jx >= 0 && jx < 32) {
                float pv = 1.f;
                if (sampled) {
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    if (j == jx) pv = xh[j];
                }
                pdtok = pv;
                have_pdtok = true;
              }
              if (lane == 0) ptx::bulk_wait_read0();
              __syncwarp();
              if (sampled) {
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                  *reinterpret_cast<float4*>(stg + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                      make_float4(xh[4 * cc], xh[4 * cc + 1], xh[4 * cc + 2], xh[4 * cc + 3]);
              } else {
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                  *reinterpret_cast<float4*>(stg + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                      make_float4(jx == 4 * cc ? 1.f : 0.f, jx == 4 * cc + 1 ? 1.f : 0.f,
                                  jx == 4 * cc + 2 ? 1.f : 0.f, jx == 4 * cc + 3 ? 1.f : 0.f);
              }
              // orders the staging writes before the TMA store and, in the first
              // half, this warp's reads of the U stage before its release
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (row0 < p.B && v0 + 32 * h < p.V) {
                  ptx::tma_store_3d(&tmPd, stg, v0 + 32 * h, s, row0, ptx::policy_evict_first());
                  ptx::bulk_commit();
                }
                if (h == 0) ptx::mbar_arrive(&emptyU[su]);
              }
            }
          }
        }
      }
      if (hasW && vrow && have_pdtok && !*abort_flag) p.pd_tok[(size_t)b * p.G + s] = pdtok;
      if (!hasS) break;  // the last sweep

      // the staging area is free for the select's scratch once this warp's
      // stores have read it; the grid barrier makes every chunk partial of
      // position q visible
      if (lane == 0) ptx::bulk_wait_read0();
      __syncwarp();
      if (!grid_barrier(p, ++nbar * (unsigned)p.n_ctas, abort_flag, s_ok, epi_tid)) {
        if (epi_tid == 0) fail();
        alive = false;
        break;
      }
      select(q);
      if (q + 1 == G && p.sel_done) {
        // every select of this CTA is done (select_rows ends with the epilogue
        // barrier): publish, then let a dependent scheduler launch
        if (epi_tid == 0) {
          __threadfence();
          atomicAdd(p.sel_done, 1u);
          ptx::launch_dependents();
        }
      }
      // E of the next sweep's S items (slot (q + 1) & 1 held E_{q-1}, whose
      // products all finished in this sweep); the gather waits for each row's
      // token, so no grid barrier follows the select: a CTA's next writes of a
      // row's partials come after it has seen the row's token, i.e. after the
      // select finished reading them
      if (q + 1 < G) {
        gather(q + 1);
      } else if (vrow) {
        // the last sweep has no S items, hence no gather: the W item's row data
        wx = token_wait(&p.tokens[(size_t)b * p.G + q], abort_flag);
        if (wx == kTokPending) fail();
        wst = __ldcg(&p.rowstat[b]);
      }
    }
    if (lane == 0) ptx::bulk_wait0();
  }

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
// Small batches (B <= nrw::NB): the same sweeps with the vocabulary on the
// MMA's M side.  A 128-request tile would carry at most NB live rows, and the
// tensor pipe would spend the sweep on the dead ones; here each product is
//     D[v, b] = sum_k W2[k, v] E[b, k]      M = 128 columns v, N = NB, K = r
// with A = the staged W2 tile (the same TMA stages, read MN-major) and B = the
// E rows in shared memory (K-major, 128-byte swizzle), so that a sweep costs
// what its W2 tiles cost to read.  TMEM lane v of an accumulator holds column
// v of the tile for every request b.  The epilogue's group 0 writes the W
// items' p_d rows (a warp stores 32 consecutive columns of a row), group 1
// forms the S items' 64-column chunk partials (warp reductions over the lanes,
// the chunk's two warps exchanging through shared memory), in the layout the
// select reads.  The select, the grid barrier and the tile claims are the
// 128-row form's.
// ---------------------------------------------------------------------------
namespace nrw {
constexpr int NB = 16;                          // batch columns of a product (M = 128 needs N % 16 == 0)
constexpr int NWS = 10;                         // W2 stages (2.5 tiles at r = 256)
constexpr int NUS = 3;                          // U stages per item
constexpr uint32_t kUStage = NB * BN * 2;       // [NB rows][128 columns] bf16, unswizzled
constexpr uint32_t kEAtom = NB / 8 * 1024;      // one 64-element K block of E: NB rows x 128 B
constexpr uint32_t kESlot = 4 * kEAtom;         // E_k for r <= 256
constexpr uint32_t kTmemCols = 4 * NB;          // two accumulators per item
constexpr uint32_t kOffE = NWS * kW2Stage;
constexpr uint32_t kOffUW = kOffE + 2 * kESlot;
constexpr uint32_t kOffUS = kOffUW + NUS * kUStage;
constexpr uint32_t kOffScr = kOffUS + NUS * kUStage;
constexpr uint32_t kScrBytes = 4096;
constexpr uint32_t kOffRow = kOffScr + kScrBytes;  // [NB] float4 (c, m, 1/S, x), [NB] gather token
constexpr uint32_t kOffXa = kOffRow + 5 * NB * 4;   // [2 buffers][2 chunks][2 halves][NB] float2
constexpr uint32_t kOffXb = kOffXa + 8 * NB * 8;    // [2][2][2][NB] float
constexpr int kRnnCols = 2;                         // state columns of a recurrent unit in this form
constexpr uint32_t kOffRnn = (kOffXb + 8 * NB * 4 + 15) / 16 * 16;  // the RNN head's unit scratch
constexpr uint32_t kOffBar = (kOffRnn + RnnUnit<kRnnCols>::kScrBytes + 63) / 64 * 64;
constexpr uint32_t kBarBytes = 1024;
constexpr size_t kSmemBytes = 1024 + kOffBar + kBarBytes;
static_assert(kSelConfOff + 2 * kTeamWarps * 4 <= (int)kScrBytes, "select scratch");
static_assert(kOffE % 1024 == 0 && kESlot % 1024 == 0 && kOffUW % 128 == 0 && kOffUS % 128 == 0, "alignment");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr int kNBars = 2 * NWS + 4 * NUS + 8 + 2 + 4 + kTQ;
static_assert(kNBars * 8 + kTQ * 4 + 16 <= (int)kBarBytes, "barrier area");
}  // namespace nrw

// Transpose-reductions over a warp of NB = 16 values per lane: each step
// halves the values a lane holds (lanes with bit `off` set keep the upper half
// and send the lower one to lane ^ off, which keeps it), so that after the
// steps at 16, 8, 4, 2 and the final exchange at 1, lanes L and L ^ 1 hold
// the reduction over all 32 lanes of value b = L >> 1.  (value, lowest index)
// argmax, and the fp32 sum in a fixed tree order.
template <int N>
__device__ __forceinline__ void halve_argmax(const float* v, const int* ix, float* vo, int* io, int off, int lane) {
  const bool hi = (lane & off) != 0;
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    float kv = hi ? v[N / 2 + j] : v[j];
    int ki = hi ? ix[N / 2 + j] : ix[j];
    const float sv = hi ? v[j] : v[N / 2 + j];
    const int si = hi ? ix[j] : ix[N / 2 + j];
    argmax_merge(kv, ki, __shfl_xor_sync(0xffffffffu, sv, off), __shfl_xor_sync(0xffffffffu, si, off));
    vo[j] = kv;
    io[j] = ki;
  }
}
__device__ __forceinline__ void xpose_argmax16(const float (&v)[16], const int (&ix)[16], float& rv, int& ri,
                                               int lane) {
  float v8[8], v4[4], v2[2], v1[1];
  int i8[8], i4[4], i2[2], i1[1];
  halve_argmax<16>(v, ix, v8, i8, 16, lane);
  halve_argmax<8>(v8, i8, v4, i4, 8, lane);
  halve_argmax<4>(v4, i4, v2, i2, 4, lane);
  halve_argmax<2>(v2, i2, v1, i1, 2, lane);
  rv = v1[0];
  ri = i1[0];
  argmax_merge(rv, ri, __shfl_xor_sync(0xffffffffu, rv, 1), __shfl_xor_sync(0xffffffffu, ri, 1));
}
template <int N>
__device__ __forceinline__ void halve_sum(const float* v, float* vo, int off, int lane) {
  const bool hi = (lane & off) != 0;
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    const float kv = hi ? v[N / 2 + j] : v[j];
    const float sv = hi ? v[j] : v[N / 2 + j];
    const float ov = __shfl_xor_sync(0xffffffffu, sv, off);
    // the lower lane's value first: both lanes of a pair add in the same order
    vo[j] = hi ? __fadd_rn(ov, kv) : __fadd_rn(kv, ov);
  }
}
__device__ __forceinline__ float xpose_sum16(const float (&v)[16], int lane) {
  float v8[8], v4[4], v2[2], v1[1];
  halve_sum<16>(v, v8, 16, lane);
  halve_sum<8>(v8, v4, 8, lane);
  halve_sum<4>(v4, v2, 4, lane);
  halve_sum<2>(v2, v1, 2, lane);
  const float o = __shfl_xor_sync(0xffffffffu, v1[0], 1);
  return (lane & 1) ? __fadd_rn(o, v1[0]) : __fadd_rn(v1[0], o);
}

// exchange point of the two warps of an S-item chunk: both arrive (lane 0,
// after the warp's shared-memory writes), then wait for the phase; bounded, so
// that a warp whose partner left on an error gives up too.  False if it gave up.
__device__ __forceinline__ bool pair_exchange(uint64_t* bar, uint32_t parity, int lane, volatile int* abort_flag) {
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(bar);
  return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, kWaitLimitNs));
}

// kRnn: the RNN head's rows (recurrent units in each gather); else W1 rows.
template <bool kRnn>
__global__ void __launch_bounds__(kThreads, 1)
    k_draft_narrow(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmW2, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int r = p.r;
  const int nkc = r / KC;
  const int G = p.G;
  const int B = p.B;
  uint8_t* sW = smem;
  uint8_t* sE = smem + nrw::kOffE;
  uint8_t* sUW = smem + nrw::kOffUW;
  uint8_t* sUS = smem + nrw::kOffUS;
  uint8_t* sScr = smem + nrw::kOffScr;
  uint8_t* sRnn = smem + nrw::kOffRnn;
  // per row: c = log2(e) / T, and the next W items' (m, 1/S, x_s) of the row
  float4* sRow = reinterpret_cast<float4*>(smem + nrw::kOffRow);
  int* sGx = reinterpret_cast<int*>(sRow + nrw::NB);
  float2* sXa = reinterpret_cast<float2*>(smem + nrw::kOffXa);
  float* sXb = reinterpret_cast<float*>(smem + nrw::kOffXb);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + nrw::kOffBar);
  uint64_t* fullW = bars;
  uint64_t* emptyW = fullW + nrw::NWS;
  uint64_t* fullUW = emptyW + nrw::NWS;
  uint64_t* emptyUW = fullUW + nrw::NUS;
  uint64_t* fullUS = emptyUW + nrw::NUS;
  uint64_t* emptyUS = fullUS + nrw::NUS;
  uint64_t* tfull = emptyUS + nrw::NUS;  // [item][buffer]
  uint64_t* tempty = tfull + 4;          // [item][buffer]
  uint64_t* eready = tempty + 4;
  uint64_t* mma_done = eready + 1;
  uint64_t* pbar = mma_done + 1;    // [step][chunk]: the S items' exchanges
  uint64_t* tqfull = pbar + 4;      // [kTQ]
  volatile int* tq = reinterpret_cast<volatile int*>(tqfull + kTQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tq) + kTQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = abort_flag + 1;
  volatile int* e_seen = s_ok + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto tile_of = [&](unsigned i, int q) {
    return i >= (unsigned)p.ntiles ? -1 : ((q & 1) ? p.ntiles - 1 - (int)i : (int)i);
  };

  if (threadIdx.x == 0) {
    for (int j = 0; j < 4; ++j) ptx::mbar_init(&pbar[j], 2);
    for (int s = 0; s < nrw::NWS; ++s) {
      ptx::mbar_init(&fullW[s], 1);
      ptx::mbar_init(&emptyW[s], 1);
    }
    for (int s = 0; s < nrw::NUS; ++s) {
      ptx::mbar_init(&fullUW[s], 1);
      ptx::mbar_init(&emptyUW[s], 4);
      ptx::mbar_init(&fullUS[s], 1);
      ptx::mbar_init(&emptyUS[s], 4);
    }
    for (int a = 0; a < 4; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 4);
    }
    ptx::mbar_init(eready, kEpiWarps);
    ptx::mbar_init(mma_done, 1);
    for (int j = 0; j < kTQ; ++j) ptx::mbar_init(&tqfull[j], 1);
    *abort_flag = 0;
    *e_seen = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, nrw::kTmemCols);
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
      // L2: a sweep's last kTailDiv-th of claims are the next sweep's first, so
      // their W2 tiles are kept (evict-last), the others read for the last time
      // in the sweep (evict-first); the S item's U rows are read again by the
      // next sweep's W item (evict-last), the W item's for the last time
      const uint64_t pol_last = ptx::policy_evict_last();
      const uint64_t pol_first = ptx::policy_evict_first();
      const unsigned tail0 = (unsigned)(p.ntiles - p.ntiles / kTailDiv);
      int iw = 0, iuw = 0, ius = 0, jq = 0;
      bool ok = true;
      for (int q = 0; q < G + p.write_pd && ok; ++q) {
        const int s = q - 1;
        const bool hasW = p.write_pd && s >= 0, hasS = s + 1 < G;
        unsigned* claim = p.sched + q;
        // the donor CTA claims nothing in the last sweep (q = G has W items only)
        const bool donate = q == G && (int)blockIdx.x == p.donor;
        unsigned ci = donate ? (unsigned)p.ntiles : atomicAdd(claim, 1u);
        int n = tile_of(ci, q);
        while (ok) {
          tq[jq % kTQ] = n;
          ptx::mbar_arrive(&tqfull[jq % kTQ]);
          ++jq;
          if (n < 0) break;
          const int v0 = n * BN;
          const bool keep = ci >= tail0;
          ci = atomicAdd(claim, 1u);
          n = tile_of(ci, q);
          for (int kc = 0; kc < nkc; ++kc, ++iw) {
            const int st = iw % nrw::NWS;
            if (!ptx::mbar_wait(&emptyW[st], ((iw / nrw::NWS) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            uint8_t* dst = sW + st * kW2Stage;
            ptx::mbar_expect_tx(&fullW[st], kW2Stage);
            for (int c = 0; c < NCH; ++c)
              ptx::tma_load_2d(dst + c * (KC * CW * 2), &tmW2, &fullW[st], v0 + c * CW, kc * KC,
                               keep ? pol_last : pol_first);
          }
          if (ok && hasW) {
            const int su = iuw % nrw::NUS;
            if (!ptx::mbar_wait(&emptyUW[su], ((iuw / nrw::NUS) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              ok = false;
            } else {
              // rows past the batch read as zeros (the box is NB rows)
              ptx::mbar_expect_tx(&fullUW[su], nrw::kUStage);
              ptx::tma_load_3d(sUW + su * nrw::kUStage, &tmU, &fullUW[su], v0, s, 0, pol_first);
              ++iuw;
            }
          }
          if (ok && hasS) {
            const int su = ius % nrw::NUS;
            if (!ptx::mbar_wait(&emptyUS[su], ((ius / nrw::NUS) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              ok = false;
            } else {
              ptx::mbar_expect_tx(&fullUS[su], nrw::kUStage);
              ptx::tma_load_3d(sUS + su * nrw::kUStage, &tmU, &fullUS[su], v0, s + 1, 0, pol_last);
              ++ius;
            }
          }
        }
      }
      if (!ok) fail();
      for (int j = max(0, iw - nrw::NWS); j < iw; ++j)
        ptx::mbar_wait(&fullW[j % nrw::NWS], (j / nrw::NWS) & 1, abort_flag, kWaitLimitNs);
      for (int j = max(0, iuw - nrw::NUS); j < iuw; ++j)
        ptx::mbar_wait(&fullUW[j % nrw::NUS], (j / nrw::NUS) & 1, abort_flag, kWaitLimitNs);
      for (int j = max(0, ius - nrw::NUS); j < ius; ++j)
        ptx::mbar_wait(&fullUS[j % nrw::NUS], (j / nrw::NUS) & 1, abort_flag, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    // The whole warp runs the loop (its values stay warp-uniform); one elected
    // lane issues the MMAs and commits.  A wait on an mbarrier queues behind
    // the shared-memory operand reads of the MMAs in flight, so a tile takes
    // all its waits (accumulators, E, W2 stages) before its first MMA and
    // then issues both products back to back; the warp takes lane 0's result
    // of each wait.
    {
      // A: W2 K-chunk [64 x 128], MN-major (the vocabulary contiguous); B: E
      // [NB x r], K-major
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, nrw::NB, true, false);
      constexpr unsigned FULL = 0xffffffffu;
      int itk[2] = {0, 0};
      int iw = 0, jq = 0;
      bool ok = true;
      auto wait0 = [&](uint64_t* bar, uint32_t parity) {
        return __shfl_sync(FULL, ptx::mbar_wait(bar, parity, abort_flag, kWaitLimitNs), 0);
      };
      auto wait_e = [&](int q) {
        if (!wait0(eready, (uint32_t)(q & 1))) return false;
        if (lane == 0) *e_seen = q + 1;
        return true;
      };
      const uint32_t sE32 = ptx::smem_u32(sE);
      for (int q = 0; q < G + p.write_pd && ok; ++q) {
        const int s = q - 1;
        const bool hasW = p.write_pd && s >= 0, hasS = s + 1 < G;
        bool e_ok = false;
        while (ok) {
          if (!wait0(&tqfull[jq % kTQ], (jq / kTQ) & 1)) {
            ok = false;
            break;
          }
          const int n = __shfl_sync(FULL, tq[jq % kTQ], 0);
          ++jq;
          if (n < 0) {
            if (hasS && !e_ok) ok = wait_e(q);
            break;
          }
          // every wait of the tile
          if (hasS && !e_ok) {
            ok = wait_e(q);
            e_ok = ok;
          }
          for (int item = 0; item < 2 && ok; ++item) {
            if (item == 0 ? !hasW : !hasS) continue;
            ok = wait0(&tempty[item * 2 + (itk[item] & 1)], ((itk[item] >> 1) & 1) ^ 1);
          }
          for (int kc = 0; kc < nkc && ok; ++kc)
            ok = wait0(&fullW[(iw + kc) % nrw::NWS], ((iw + kc) / nrw::NWS) & 1);
          if (!ok) break;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
            for (int item = 0; item < 2; ++item) {
              if (item == 0 ? !hasW : !hasS) continue;
              const int ab = item * 2 + (itk[item] & 1);
              const int kk = item == 0 ? s : s + 1;
              const uint32_t eb = sE32 + (uint32_t)(kk & 1) * nrw::kESlot;
              const uint32_t d = tmem + (uint32_t)(ab * nrw::NB);
              for (int kc = 0; kc < nkc; ++kc) {
                const uint32_t aW2 = ptx::smem_u32(sW + ((iw + kc) % nrw::NWS) * kW2Stage);
#pragma unroll
                for (int k4 = 0; k4 < KC / 16; ++k4) {
                  // A: two 64-column blocks 8 KB apart, 8-row K groups 1024 B
                  //    apart; B: E's K block kc, 16 elements (32 B) per step
                  const uint64_t ad = ptx::smem_desc_sw128(aW2 + k4 * 2048, KC * CW * 2, 1024);
                  const uint64_t bd = ptx::smem_desc_sw128(eb + (uint32_t)kc * nrw::kEAtom + k4 * 32, 16, 1024);
                  ptx::tc_mma(d, ad, bd, idesc, (kc | k4) > 0 ? 1u : 0u);
                }
              }
              ptx::tc_commit(&tfull[ab]);
            }
            // the tile's W2 stages are free once both of its products are done
            for (int kc = 0; kc < nkc; ++kc) ptx::tc_commit(&emptyW[(iw + kc) % nrw::NWS]);
          }
          __syncwarp();
          if (hasW) ++itk[0];
          if (hasS) ++itk[1];
          iw += nkc;
        }
      }
      if (!ok && lane == 0) fail();
      if (ptx::elect_one()) ptx::tc_commit(mma_done);
      __syncwarp();
      wait0(mma_done, 0);
    }
  } else {
    // ------------------------------ epilogue ----------------------------------
    const int ew = warp - kEpiWarp0;
    const int epi_tid = ew * 32 + lane;
    const int g = ew >> 2;       // 0: W items, 1: S items
    const int qd = warp & 3;     // TMEM lanes 32 qd .. 32 qd + 31: columns of the tile
    const int ch = qd >> 1;      // the 64-column chunk of those columns
    const int half = qd & 1;     // this warp's half of the chunk
    const uint32_t lane_bits = (uint32_t)(qd * 32) << 16;
    const int team = ew / kTeamWarps, tw = ew % kTeamWarps;
    unsigned nbar = 0;
    int jq = 0, itw = 0, its = 0, iuw = 0, ius = 0, ix = 0;
    bool alive = true;

    // bit b: row b is sampled (T > 0); the others are greedy
    uint32_t samp = 0u;
    for (int b = 0; b < B; ++b) samp |= (p.temp[b] > 0.f ? 1u : 0u) << b;
    if (epi_tid < B) sRow[epi_tid] = make_float4(row_scale(p.temp[epi_tid]), 0.f, 1.f, 0.f);
    // both E slots zero: the rows past the batch stay so (their products fill
    // accumulator columns nobody reads)
    for (int i = epi_tid; i < (int)(2 * nrw::kESlot / 16); i += kEpiThreads)
      reinterpret_cast<uint4*>(sE)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int rb = (int)blockIdx.x + p.n_ctas * ew; rb < B; rb += p.n_ctas * kEpiWarps)
      for (int k = lane; k < G; k += 32) p.tokens[(size_t)rb * G + k] = kTokPending;
    epi_sync();

    // E_k = W1[x_{k-1}] (x_0 = anchor) of every row into slot k & 1, and for
    // k >= 1 the next W items' row data: x_{k-1} and (m, S) of position k - 1
    auto gather = [&](int k) {
      if (epi_tid < B) {
        const int b = epi_tid;
        int x;
        if (k == 0) {
          x = p.anchor[b];
        } else {
          x = token_wait(&p.tokens[(size_t)b * G + k - 1], abort_flag);
          if (x == kTokPending) {
            fail();
            x = 0;
          }
          const float2 st = __ldcg(&p.rowstat[b]);
          sRow[b].y = st.x;
          sRow[b].z = inv_sum(st.y);
          sRow[b].w = __int_as_float(x);
        }
        if (x < 0 || x >= p.V) {
          report_error(p.hdr, DSPARK_BAD_INPUT, x);
          x = 0;
        }
        sGx[b] = x;
      }
      epi_sync();
      if constexpr (kRnn) {
        // the recurrent units of position k, then E_k once every unit (one
        // row block: B <= 16) has finished
        if (!rnn_units<nrw::kRnnCols>(p, k, sRnn, epi_tid, abort_flag)) fail();
        if (epi_tid == 0) {
          const unsigned target = (unsigned)(r / nrw::kRnnCols);
          const unsigned* cnt = p.rnn_done + (size_t)k * p.n_mtiles;
          int okw = *abort_flag ? 0 : 1;
          const uint64_t t0 = ptx::globaltimer_ns();
          while (okw && ld_acquire(cnt) < target) {
            if (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitLimitNs) okw = 0;
            __nanosleep(32);
          }
          *s_ok = okw;
        }
        epi_sync();
        if (!*s_ok && epi_tid == 0) fail();
      }
      // row b's r / 8 16-byte pieces; piece j holds K elements 8 j .. 8 j + 7:
      // K block j / 8, 16-byte column (j % 8) ^ (b % 8) of the row's 128 bytes
      uint8_t* slot = sE + (k & 1) * nrw::kESlot;
      const int per = r / 8;
      for (int i = epi_tid; i < B * per; i += kEpiThreads) {
        const int b = i / per, j = i - b * per;
        // (L2 for the RNN head's rows: written during this launch)
        const uint4 v = kRnn ? __ldcg(reinterpret_cast<const uint4*>(p.rnn_E + ((size_t)(k & 1) * B + b) * r) + j)
                             : __ldg(reinterpret_cast<const uint4*>(p.W1 + (size_t)sGx[b] * r) + j);
        *reinterpret_cast<uint4*>(slot + (j >> 3) * nrw::kEAtom + (b >> 3) * 1024 + (b & 7) * 128 +
                                  (((j & 7) ^ (b & 7)) << 4)) = v;
      }
      // the MMA reads the slot through the async proxy
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (*e_seen < k) {
          if (*abort_flag || ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            fail();
            break;
          }
          __nanosleep(32);
        }
        ptx::mbar_arrive(eready);
      }
    };

    if (!*abort_flag) gather(0);
    for (int q = 0; q < G + p.write_pd && alive; ++q) {
      const int s = q - 1;
      const bool hasW = p.write_pd && s >= 0, hasS = s + 1 < G;
      const bool mine = g == 0 ? hasW : hasS;
      bool tiles_ok = true;
      while (tiles_ok) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&tqfull[jq % kTQ], (jq / kTQ) & 1, abort_flag, kWaitLimitNs))) {
          if (lane == 0) fail();
          tiles_ok = false;
          break;
        }
        const int n = tq[jq % kTQ];
        ++jq;
        if (n < 0) break;
        if (!mine) continue;
        const int col = 32 * qd + lane;  // this lane's column of the tile
        const int vt = n * BN + col;
        const bool vin = vt < p.V;
        // the accumulator and the U stage of this warp's item
        int& it = g == 0 ? itw : its;
        int& iu = g == 0 ? iuw : ius;
        const int ab = g * 2 + (it & 1);
        const int su = iu % nrw::NUS;
        uint64_t* fullU = g == 0 ? fullUW : fullUS;
        uint64_t* emptyU = g == 0 ? emptyUW : emptyUS;
        bool ok = ptx::mbar_wait(&tfull[ab], (it >> 1) & 1, abort_flag, kWaitLimitNs);
        if (ok) ok = ptx::mbar_wait(&fullU[su], (iu / nrw::NUS) & 1, abort_flag, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) fail();
          tiles_ok = false;
          break;
        }
        ++it;
        ++iu;
        ptx::tc_fence_after();
        float acc[nrw::NB];
        __syncwarp();
        ptx::tmem_ld16(tmem + lane_bits + (uint32_t)(ab * nrw::NB), acc);
        const __nv_bfloat16* ur =
            reinterpret_cast<const __nv_bfloat16*>((g == 0 ? sUW : sUS) + su * nrw::kUStage) + col;
        float l[nrw::NB];
#pragma unroll
        for (int b = 0; b < nrw::NB; ++b) l[b] = b < B ? __bfloat162float(ur[b * BN]) : 0.f;
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        // the U stage's next fill is an async-proxy write: order the reads first
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&tempty[ab]);
          ptx::mbar_arrive(&emptyU[su]);
        }
#pragma unroll
        for (int b = 0; b < nrw::NB; ++b) l[b] = add_base(l[b], acc[b]);
        if (g == 0) {
          // W item: p_d^s = 2^(l c - m) / S, one-hot for greedy rows
#pragma unroll
          for (int b = 0; b < nrw::NB; ++b) {
            if (b >= B) break;
            const float4 rw = sRow[b];
            const int xs = __float_as_int(rw.w);
            const float pw = __fmul_rn(exp_scaled(l[b], rw.x, rw.y), rw.z);
            const float pv = ((samp >> b) & 1u) ? pw : (vt == xs ? 1.f : 0.f);
            // streaming store (read once, by verify)
            if (vin) __stcs(p.pd_rows + ((size_t)b * G + s) * p.V + vt, pv);
            if (vt == xs) p.pd_tok[(size_t)b * G + s] = pv;
          }
        } else {
          // S item: chunk partials of position s + 1.  Step 1: each warp's
          // (value, lowest index) argmax of the logits over its 32 columns, for
          // every row at once (a sampled row takes the value: the max of l c
          // is at the max of l for c > 0)
          const int buf = ix & 1;
          ++ix;
          float2* xa = sXa + (size_t)((buf * 2 + ch) * 2) * nrw::NB;
          float* xb = sXb + (size_t)((buf * 2 + ch) * 2) * nrw::NB;
          const int bl = lane >> 1;  // the row whose reductions this lane ends with
          {
            int li[nrw::NB];
#pragma unroll
            for (int b = 0; b < nrw::NB; ++b) {
              li[b] = (vin && b < B) ? vt : INT_MAX;
              if (!(vin && b < B)) l[b] = -INFINITY;
            }
            float rv;
            int ri;
            xpose_argmax16(l, li, rv, ri, lane);
            if (!(lane & 1) && bl < B) xa[half * nrw::NB + bl] = make_float2(rv, __int_as_float(ri));
          }
          if (!pair_exchange(&pbar[ch], (uint32_t)buf, lane, abort_flag)) {
            if (lane == 0) fail();
            tiles_ok = false;
            break;
          }
          // step 2: the chunk max of each sampled row, then each warp's sum of
          // 2^(l c - m_chunk) for every row at once
          {
            float e[nrw::NB];
#pragma unroll
            for (int b = 0; b < nrw::NB; ++b) {
              e[b] = 0.f;
              if (b < B && ((samp >> b) & 1u)) {
                const float lm = fmaxf(xa[b].x, xa[nrw::NB + b].x);
                const float cb = sRow[b].x;
                // (l is -inf past V: those columns weigh nothing)
                if (lm != -INFINITY) e[b] = exp_scaled(l[b], cb, scale_logit(lm, cb));
              }
            }
            const float ws = xpose_sum16(e, lane);
            if (!(lane & 1) && bl < B) xb[half * nrw::NB + bl] = ws;
          }
          if (!pair_exchange(&pbar[2 + ch], (uint32_t)buf, lane, abort_flag)) {
            if (lane == 0) fail();
            tiles_ok = false;
            break;
          }
          const int j = n * NCH + ch;  // the chunk's index in the row
          if (half == 0 && lane < B && j * CW < p.V) {
            const int b = lane;
            float2 part;
            if ((samp >> b) & 1u) {
              const float lm = fmaxf(xa[b].x, xa[nrw::NB + b].x);
              part = lm == -INFINITY ? make_float2(-INFINITY, 0.f)
                                     : make_float2(scale_logit(lm, sRow[b].x), __fadd_rn(xb[b], xb[nrw::NB + b]));
            } else {
              float v = xa[b].x;
              int i = __float_as_int(xa[b].y);
              argmax_merge(v, i, xa[nrw::NB + b].x, __float_as_int(xa[nrw::NB + b].y));
              part = make_float2(v, __int_as_float(i));
            }
            // (a small batch's partials stay in L2 without a policy)
            p.part[(size_t)b * p.pstride + (j % p.ept) * 128 + j / p.ept] = part;
          }
        }
      }
      if (!hasS) break;  // the last sweep
      if (!grid_barrier(p, ++nbar * (unsigned)p.n_ctas, abort_flag, s_ok, epi_tid)) {
        if (epi_tid == 0) fail();
        alive = false;
        break;
      }
      select_rows(p, q, sScr, team, tw, lane);
      if (q + 1 == G && p.sel_done && epi_tid == 0) {
        // every select of this CTA is done: publish, then let a dependent
        // scheduler launch (as in the 128-row form)
        __threadfence();
        atomicAdd(p.sel_done, 1u);
        ptx::launch_dependents();
      }
      if (q + 1 < G) {
        gather(q + 1);
      } else {
        // the last sweep has no S items, hence no gather: the W items' row data
        if (epi_tid < B) {
          const int b = epi_tid;
          int x = token_wait(&p.tokens[(size_t)b * G + q], abort_flag);
          if (x == kTokPending) {
            fail();
            x = 0;
          }
          const float2 st = __ldcg(&p.rowstat[b]);
          sRow[b].y = st.x;
          sRow[b].z = inv_sum(st.y);
          sRow[b].w = __int_as_float(x);
        }
        epi_sync();
      }
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, nrw::kTmemCols);
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
                   const cuuint64_t* strides, const cuuint32_t* box,
                   CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The small-batch form runs for B <= nrw::NB unless DSPARK_DRAFT_FORM=wide
// asks for the 128-row form at every batch.
static bool narrow_enabled() {
  static int on = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* e = getenv("DSPARK_DRAFT_FORM");
    on = (e && std::string(e) == "wide") ? 0 : 1;
  });
  return on != 0;
}

// The 128-row form's stage rings for a batch of n_mtiles M-tiles;
// DSPARK_FUSED_RING=w2 or =u picks one at every batch.
static bool ring_w2_deep(int n_mtiles) {
  static int force = -1;  // -1: by the batch, 0: U-deep, 1: W2-deep
  static std::once_flag once;
  std::call_once(once, [] {
    const char* e = getenv("DSPARK_FUSED_RING");
    if (e && std::string(e) == "w2") force = 1;
    if (e && std::string(e) == "u") force = 0;
  });
  return force >= 0 ? force == 1 : n_mtiles <= kRingW2DeepMaxMtiles;
}

}  // namespace fz

// The fused-sweep kernel needs every CTA resident (cooperative launch, one
// CTA per SM) and at most one CTA's worth of M-tiles per SM; returns
// cudaErrorNotSupported when it cannot run, so that the caller falls back.
cudaError_t launch_draft_fused(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s,
                               DraftOverlap* ov) {
  const dspark_dims& d = a.dims;
  int dev = 0, sms = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorNotSupported;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  const int n_mtiles = (d.B + fz::BM - 1) / fz::BM;
  if (!coop || sms <= 0 || n_mtiles > sms || d.r > 2 * (int)fz::kESlotCols || (d.r % (8 * 8)) != 0)
    return cudaErrorNotSupported;
  const cuuint64_t V = (cuuint64_t)d.V, G = (cuuint64_t)d.gamma, B = (cuuint64_t)d.B, r = (cuuint64_t)d.r;
  // small batches: the vocabulary on the MMA's M side (k_draft_narrow)
  const bool narrow = d.B <= fz::nrw::NB && fz::narrow_enabled();
  // the RNN head runs with p_d rows and reads W_rnn rows with 16-byte loads
  const bool rnn = a.head == DSPARK_HEAD_RNN;
  if (rnn && (!a.pd_rows || !a.W_rnn || (reinterpret_cast<uintptr_t>(a.W_rnn) % 16) != 0 ||
              ((2 * d.r + d.H) % 8) != 0))
    return cudaErrorNotSupported;
  CUtensorMap tmU, tmW2, tmPd = {};  // tmPd stays unused without p_d rows and in the small-batch form
  if (narrow) {
    // U rows of all requests of one position, 128 columns, unswizzled
    const cuuint64_t dims[3] = {V, G, B};
    const cuuint64_t strides[2] = {V * 2, G * V * 2};
    const cuuint32_t box[3] = {fz::BN, 1, fz::nrw::NB};
    if (!fz::encode(&tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.U, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    const cuuint64_t dims[3] = {V, G, B};
    const cuuint64_t strides[2] = {V * 2, G * V * 2};
    const cuuint32_t box[3] = {fz::CW, 1, fz::BM};
    if (!fz::encode(&tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.U, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {V, r};
    const cuuint64_t strides[1] = {V * 2};
    const cuuint32_t box[2] = {fz::CW, fz::KC};
    if (!fz::encode(&tmW2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {V, G, B};
    const cuuint64_t strides[2] = {V * 4, G * V * 4};
    const cuuint32_t box[3] = {32, 1, 32};
    if (!narrow && a.pd_rows && !fz::encode(&tmPd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.pd_rows, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  const bool w2deep = fz::ring_w2_deep(n_mtiles);
  const void* kfn =
      narrow ? (rnn ? (const void*)fz::k_draft_narrow<true> : (const void*)fz::k_draft_narrow<false>)
      : w2deep ? (rnn ? (const void*)fz::k_draft_fused<true, fz::kRingW2Deep>
                      : (const void*)fz::k_draft_fused<false, fz::kRingW2Deep>)
               : (rnn ? (const void*)fz::k_draft_fused<true, fz::kRingUDeep>
                      : (const void*)fz::k_draft_fused<false, fz::kRingUDeep>);
  const size_t smem = narrow ? fz::nrw::kSmemBytes : fz::smem_bytes(w2deep ? fz::kRingW2Deep : fz::kRingUDeep);
  if (const cudaError_t ae = ensure_smem_limit(kfn, (int)smem); ae != cudaSuccess) return ae;

  fz::Params p;
  p.B = d.B;
  p.G = d.gamma;
  p.V = d.V;
  p.r = d.r;
  p.H = d.H;
  p.seed = a.seed;
  p.ntiles = (d.V + fz::BN - 1) / fz::BN;
  p.nparts = (d.V + fz::CW - 1) / fz::CW;
  p.ctas_per_m = std::max(1, std::min(p.ntiles, sms / n_mtiles));
  p.n_ctas = n_mtiles * p.ctas_per_m;
  p.n_mtiles = n_mtiles;
  p.ept = (p.nparts + fz::kTeamWarps * 32 - 1) / (fz::kTeamWarps * 32);
  p.pstride = p.ept * fz::kTeamWarps * 32;
  if (p.ept > fz::kMaxE) return cudaErrorNotSupported;
  p.U = static_cast<const __nv_bfloat16*>(a.U);
  p.W1 = static_cast<const __nv_bfloat16*>(a.W1);
  p.W2 = static_cast<const __nv_bfloat16*>(a.W2);
  p.w = static_cast<const __nv_bfloat16*>(a.w);
  p.h = static_cast<const __nv_bfloat16*>(a.h);
  p.anchor = a.anchor;
  p.temp = a.temp;
  p.req_id = a.req_id;
  p.rowstat = reinterpret_cast<float2*>(ws + L.rowstat);
  p.tokens = a.tokens;
  p.part = reinterpret_cast<float2*>(ws + L.part);
  p.pd_tok = a.pd_tok;
  p.pd_rows = a.pd_rows;
  p.write_pd = a.pd_rows ? 1 : 0;
  p.pd_stat = reinterpret_cast<float2*>(a.pd_stat);
  p.conf_logit = a.conf_logit;
  p.conf = a.conf;
  p.gbar = reinterpret_cast<unsigned*>(ws + L.gbar);
  p.sched = reinterpret_cast<unsigned*>(ws + L.gbar + 16);
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.W_rnn = nullptr;
  p.rnn_P = nullptr;
  p.rnn_S = nullptr;
  p.rnn_E = nullptr;
  p.rnn_done = p.sched + (size_t)(d.gamma + 1) * n_mtiles;
  // a scheduler behind this launch: either form with p_d rows (a last sweep
  // to run beside) and more than one CTA.  It needs a free SM: a donor CTA
  // when the grid fills every SM; otherwise an idle SM takes it and every CTA
  // keeps its share of the last sweep (a donor would leave its M-tile one CTA
  // short for that sweep).
  p.sel_done = nullptr;
  p.donor = -1;
  if (ov && ov->want && a.pd_rows && p.n_ctas > 1) {
    p.sel_done = p.gbar + 1;  // in the counters' 16-byte head, zeroed below
    p.donor = p.n_ctas < sms ? -1 : p.n_ctas - 1;
  }
  if (rnn) {
    // the h part of every position's projection, one GEMM before the sweeps
    float* P = reinterpret_cast<float*>(ws + L.rnn_p);
    if (d.H > 0) {
      const cudaError_t he = launch_rnn_hproj(a, P, reinterpret_cast<WsHeader*>(ws), s);
      if (he != cudaSuccess) return he;
      p.rnn_P = P;
    }
    p.W_rnn = static_cast<const __nv_bfloat16*>(a.W_rnn);
    p.rnn_S = reinterpret_cast<float*>(ws + L.rnn_s);
    p.rnn_E = reinterpret_cast<__nv_bfloat16*>(ws + L.E);
  }
  // the grid-barrier counter, the tile claims of every sweep and the
  // recurrent-unit counters of every position
  cudaError_t e = cudaMemsetAsync(p.gbar, 0, 16 + sizeof(unsigned) * (size_t)(2 * d.gamma + 1) * n_mtiles, s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_ctas);
  cfg.blockDim = dim3(fz::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  if (narrow)
    e = rnn ? cudaLaunchKernelEx(&cfg, fz::k_draft_narrow<true>, tmU, tmW2, p)
            : cudaLaunchKernelEx(&cfg, fz::k_draft_narrow<false>, tmU, tmW2, p);
  else if (w2deep)
    e = rnn ? cudaLaunchKernelEx(&cfg, fz::k_draft_fused<true, fz::kRingW2Deep>, tmU, tmW2, tmPd, p)
            : cudaLaunchKernelEx(&cfg, fz::k_draft_fused<false, fz::kRingW2Deep>, tmU, tmW2, tmPd, p);
  else
    e = rnn ? cudaLaunchKernelEx(&cfg, fz::k_draft_fused<true, fz::kRingUDeep>, tmU, tmW2, tmPd, p)
            : cudaLaunchKernelEx(&cfg, fz::k_draft_fused<false, fz::kRingUDeep>, tmU, tmW2, tmPd, p);
  if (e == cudaSuccess && p.sel_done) {
    ov->armed = true;
    ov->sel_done = p.sel_done;
    ov->n_ctas = (unsigned)p.n_ctas;
  }
  return e;
}

}  // namespace dspark
