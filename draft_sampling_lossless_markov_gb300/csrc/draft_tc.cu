// Tensor-core (tcgen05) logits passes of the draft sampler, sm_103a.
//
// The Markov-head bias of position k is a dense contraction
//     bias[b, v] = E[b, :] . W2[:, v],   E[b] = W1[x_{k-1}]      (B x r x V)
// ([DSpark] 方法细节, "马尔可夫头（Markov head）的实现").  With r = 256 it is
// 2 r = 512 flop per (b, v) against 6 bytes of U read + p_d write, i.e. far
// above the CUDA-core ridge, so it runs on the 5th-generation tensor cores.
//
// Tile: 128 requests (TMEM lanes) x 192 vocabulary columns, K = r.  One
// tcgen05.mma instruction costs about the same for N = 64 and N = 128 and
// reaches the tensor-core peak only near N = 256, so the tile is as wide as
// TMEM allows: E (the A operand, r/2 columns) plus two 192-column fp32
// accumulators fill the 512 columns.
//
//   warp 0    TMA producer, two rings: W2 in K-chunks [64 x 192] (L2
//             evict-last: every pass re-reads W2) and U in column chunks
//             [128 x 64] (L2 evict-first: streamed), all 128B-swizzled
//   warp 1    allocates TMEM, issues tcgen05.mma (A = E from TMEM, B = W2
//             K-chunk from shared memory, MN-major, N = 192) into one of the
//             two accumulators, commits to mbarriers
//   warps 2-13 epilogue, three groups of four warps (one per TMEM lane
//             quarter); group g owns the g-th 64-column chunk of every tile, so
//             all three work on a tile at once.  The groups first copy the E
//             rows into TMEM.  Per tile: TMEM -> registers, + U, then either
//             the chunk's (max, sum, argmax) partial (pass 1) or the
//             probability row p_d = 2^(y - m) / S written through a per-warp
//             swizzled staging buffer with TMA stores (pass 2)
//
// A CTA owns one 128-row M-tile; the vocabulary tiles of an M-tile are dealt
// round-robin to its CTAs.  Every mbarrier wait gives up after two seconds: the
// kernel then records DSPARK_TIMEOUT in the workspace error word, lets the
// other roles leave their loops, waits for its own TMA loads and stores, frees
// its TMEM and returns.
#include <cuda.h>

#include <cstdlib>
#include <mutex>
#include <string>

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
constexpr int kThreads = 64 + kGroups * 128;         // producer, MMA, epilogue
constexpr int kEpiWarps = kGroups * 4;
constexpr int kEpiWarp0 = 2;
constexpr int kStagingPerWarp = 32 * 32 * 4;         // [32 rows x 32 cols] fp32
constexpr uint32_t kW2Stage = KC * BN * 2;           // 24 KB
constexpr uint32_t kUStage = BM * CW * 2;            // 16 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol0 = 128;                   // accumulators after the E columns

struct Params {
  int B, G, V, r, H, k, ntiles, nparts, ctas_per_m;
  int m_first;   // first M-tile of this launch
  int u_keep;    // pass 1 loads U evict-last: pass 2 of the same rows follows at once
  const __nv_bfloat16* W1;   // [V, r]
  const __nv_bfloat16* w;    // [H + r] confidence weight (w_e = w + H)
  const float* zh;           // [B, G] w_h . h
  const int32_t* anchor;     // [B]
  const float* temp;
  const float2* rowstat;     // [B] (m, S) of position k (pass 2)
  const float4* sel;         // [B] crossing chunk, prefix, target, hit (pass 2)
  int32_t* tokens;           // [B, G]
  float4* part;              // [B, nparts] per 64-column chunk (pass 1)
  float* pd_tok;
  float* conf_logit;
  float* conf;
  WsHeader* hdr;
};

__host__ __device__ constexpr int w2_stages(bool write) { return write ? 3 : 4; }
__host__ __device__ constexpr int u_stages(bool write) { return write ? 5 : 6; }

__host__ __device__ inline size_t smem_bytes(bool write) {
  const size_t staging = write ? (size_t)kEpiWarps * kStagingPerWarp : 0;
  return 1024 + w2_stages(write) * (size_t)kW2Stage + u_stages(write) * (size_t)kUStage + staging + 512;
}

template <bool WRITE>
__global__ void __launch_bounds__(kThreads, 1)
    k_logits_tc(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmW2,
                const __grid_constant__ CUtensorMap tmPd, Params p) {
  constexpr int NW = w2_stages(WRITE);
  constexpr int NU = u_stages(WRITE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int r = p.r;
  const int nkc = r / KC;  // K-chunks per tile
  uint8_t* sW = smem;
  uint8_t* sU = sW + NW * kW2Stage;
  uint8_t* sStg = sU + NU * kUStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + (WRITE ? kEpiWarps * kStagingPerWarp : 0));
  uint64_t* fullW = bars;
  uint64_t* emptyW = fullW + NW;
  uint64_t* fullU = emptyW + NW;
  uint64_t* emptyU = fullU + NU;
  uint64_t* tfull = emptyU + NU;
  uint64_t* tempty = tfull + 2;
  uint64_t* eready = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(eready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = p.m_first + (int)blockIdx.x / p.ctas_per_m;
  // vocabulary tiles of this M-tile are dealt round-robin, so that all CTAs
  // sweep the vocabulary together.  Pass 1 sweeps it upward and pass 2
  // downward: pass 2 then starts on the tiles pass 1 touched last, whose U and
  // W2 lines are the likeliest to still be in L2 (the next position's pass 1
  // again starts where pass 2 ended).
  const int n_lo = blockIdx.x % p.ctas_per_m;
  const int stride = p.ctas_per_m;
  const int count = n_lo < p.ntiles ? (p.ntiles - n_lo + stride - 1) / stride : 0;
  auto tile_of = [&](int i) { return n_lo + (WRITE ? count - 1 - i : i) * stride; };
  const int row_base = m_tile * BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NW; ++s) {
      ptx::mbar_init(&fullW[s], 1);
      ptx::mbar_init(&emptyW[s], 1);
    }
    for (int s = 0; s < NU; ++s) {
      ptx::mbar_init(&fullU[s], 1);
      ptx::mbar_init(&emptyU[s], 4);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], kEpiWarps);
    }
    ptx::mbar_init(eready, kEpiWarps);
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

  if (count > 0 && warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      const uint64_t pol_last = ptx::policy_evict_last();
      const uint64_t pol_first = ptx::policy_evict_first();
      const uint64_t pol_u = (!WRITE && p.u_keep) ? pol_last : pol_first;
      int iw = 0, iu = 0;  // items issued into each ring
      bool ok = true;
      for (int i = 0; i < count && ok; ++i) {
        const int v0 = tile_of(i) * BN;
        for (int kc = 0; kc < nkc && ok; ++kc, ++iw) {
          const int s = iw % NW;
          if (!ptx::mbar_wait(&emptyW[s], ((iw / NW) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          uint8_t* st = sW + s * kW2Stage;
          ptx::mbar_expect_tx(&fullW[s], kW2Stage);
          for (int c = 0; c < NCH; ++c)
            ptx::tma_load_2d(st + c * (KC * CW * 2), &tmW2, &fullW[s], v0 + c * CW, kc * KC, pol_last);
        }
        for (int c = 0; c < NCH && ok; ++c, ++iu) {
          const int s = iu % NU;
          if (!ptx::mbar_wait(&emptyU[s], ((iu / NU) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::mbar_expect_tx(&fullU[s], kUStage);
          ptx::tma_load_3d(sU + s * kUStage, &tmU, &fullU[s], v0 + c * CW, p.k, row_base, pol_u);
        }
      }
      if (!ok) fail();
      // every load this thread issued has landed before the CTA may exit
      for (int j = max(0, iw - NW); j < iw; ++j) ptx::mbar_wait(&fullW[j % NW], (j / NW) & 1, abort_flag, kWaitLimitNs);
      for (int j = max(0, iu - NU); j < iu; ++j) ptx::mbar_wait(&fullU[j % NU], (j / NU) & 1, abort_flag, kWaitLimitNs);
    }
  } else if (count > 0 && warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, false, true);
      int issued = 0, iw = 0;
      bool ok = ptx::mbar_wait(eready, 0, abort_flag, kWaitLimitNs);
      if (ok) ptx::tc_fence_after();
      for (int i = 0; i < count && ok; ++i) {
        const int a = i & 1;
        if (!ptx::mbar_wait(&tempty[a], ((i >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + kAccCol0 + (uint32_t)(a * BN);
        for (int kc = 0; kc < nkc; ++kc, ++iw) {
          const int s = iw % NW;
          if (!ptx::mbar_wait(&fullW[s], (iw / NW) & 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t aW2 = ptx::smem_u32(sW + s * kW2Stage);
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
        issued = i + 1;
      }
      if (!ok) fail();
      // the last commit tracks every MMA issued: TMEM is not freed under a running MMA
      if (issued > 0)
        ptx::mbar_wait(&tfull[(issued - 1) & 1], ((issued - 1) >> 1) & 1, abort_flag, kWaitLimitNs);
    }
  } else if (count > 0 && warp >= kEpiWarp0) {
    // ------------------------------ epilogue ----------------------------------
    const int g = (warp - kEpiWarp0) >> 2;  // group: tiles i with i % 2 == g
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;          // row within the M-tile
    const int b = row_base + row;
    const bool vrow = b < p.B;
    const uint32_t lane_bits = (uint32_t)(q * 32) << 16;
    const int npieces = r / 64;  // 64-element pieces of an E row (32 TMEM columns each)
    {
      // E = W1[x_{k-1}] (x_0 = anchor) into TMEM columns [0, r/2): two bf16 per
      // column, zeros past B.  Group g copies pieces g and g + 3 of its rows, so
      // every load of a row is in flight at once before the first MMA may start.
      int x = 0;
      if (vrow) {
        x = (p.k == 0) ? p.anchor[b] : p.tokens[(size_t)b * p.G + p.k - 1];
        if (x < 0 || x >= p.V) {
          if (g == 0) report_error(p.hdr, DSPARK_BAD_INPUT, x);
          x = 0;
        }
      }
      const uint4* src = reinterpret_cast<const uint4*>(p.W1 + (size_t)x * r);
      uint32_t wv[2][32];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int pc = g + kGroups * s;
        if (pc < npieces) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint4 qv = vrow ? src[pc * 8 + e] : make_uint4(0u, 0u, 0u, 0u);
            wv[s][4 * e] = qv.x;
            wv[s][4 * e + 1] = qv.y;
            wv[s][4 * e + 2] = qv.z;
            wv[s][4 * e + 3] = qv.w;
          }
        }
      }
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int pc = g + kGroups * s;
        if (pc < npieces) ptx::tmem_st32(tmem + lane_bits + (uint32_t)(pc * 32), wv[s]);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(eready);
    }
    if (!WRITE && g == 0 && n_lo == 0) {
      // pass 1 on the first CTA of the M-tile also forms the confidence of
      // position k: z = w_h . h_k + w_e . W1[x_{k-1}], reading the E row back
      // from TMEM once every group has stored its pieces
      bool ok = ptx::mbar_wait(eready, 0, abort_flag, kWaitLimitNs);
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
          const float z = p.zh[(size_t)b * p.G + p.k] + zacc;
          p.conf_logit[(size_t)b * p.G + p.k] = z;
          p.conf[(size_t)b * p.G + p.k] = 1.f / (1.f + expf(-z));
        }
      } else if (lane == 0) {
        fail();
      }
    }

    const float T_ = vrow ? p.temp[b] : 1.f;
    const bool sampled = T_ > 0.f;
    const float c = row_scale(T_);
    float rm = 0.f, rinvS = 1.f;
    int xb = -1;          // greedy rows: the token chosen by the select kernel
    int cstar = -1;       // sampled rows: the 64-column chunk that holds the draw
    float sbase = 0.f, starget = 0.f;
    bool shit = false;
    if (WRITE && vrow) {
      const float2 st = p.rowstat[b];
      rm = st.x;
      rinvS = inv_sum(st.y);
      if (sampled) {
        const float4 sv = p.sel[b];
        cstar = __float_as_int(sv.x);
        sbase = sv.y;
        starget = sv.z;
        shit = __float_as_int(sv.w) != 0;
      } else {
        xb = p.tokens[(size_t)b * p.G + p.k];
      }
    }
    uint8_t* stg = sStg + (warp - kEpiWarp0) * kStagingPerWarp;
    float pdtok = 0.f;
    bool have_pdtok = false;
    const int ch = g;  // the chunk of every tile this group owns
    for (int i = 0; i < count; ++i) {
      const int a = i & 1;
      const int n = tile_of(i);
      const int v0 = n * BN + ch * CW;
      bool ok = ptx::mbar_wait(&tfull[a], (i >> 1) & 1, abort_flag, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) fail();
        break;
      }
      ptx::tc_fence_after();
      float acc[64];
      {
        float h0[32], h1[32];
        const uint32_t ta = tmem + lane_bits + kAccCol0 + (uint32_t)(a * BN + ch * CW);
        ptx::tmem_ld32(ta, h0);
        ptx::tmem_ld32(ta + 32, h1);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          acc[j] = h0[j];
          acc[32 + j] = h1[j];
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[a]);
      const int iu = i * NCH + ch, su = iu % NU;
      ok = ptx::mbar_wait(&fullU[su], (iu / NU) & 1, abort_flag, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) fail();
        break;
      }
      {
        // U row of this thread: 8 swizzled 16-byte chunks of 8 bf16
        const uint8_t* su_row = sU + su * kUStage + row * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint4 qv = *reinterpret_cast<const uint4*>(su_row + ((cc ^ (row & 7)) << 4));
          const __nv_bfloat162* bp = reinterpret_cast<const __nv_bfloat162*>(&qv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(bp[e]);
            acc[8 * cc + 2 * e] = add_base(f.x, acc[8 * cc + 2 * e]);
            acc[8 * cc + 2 * e + 1] = add_base(f.y, acc[8 * cc + 2 * e + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&emptyU[su]);
      // acc[j] now holds the logit l of column v0 + j; columns past V are masked
      const int nvalid = min(CW, p.V - v0);
      if (!WRITE) {
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          acc[j] = (j < nvalid) ? scale_logit(acc[j], c) : -INFINITY;  // y = l c (greedy rows: c = 1)
          mx[j & 3] = fmaxf(mx[j & 3], acc[j]);
        }
        const float mc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        float sm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 64; ++j) sm[j & 3] += exp_shifted(acc[j], mc);
        float av = -INFINITY;
        int ai = INT_MAX;
        if (!sampled) {
          // greedy: argmax of y = l, ties to the lowest column
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (acc[j] > av) {
              av = acc[j];
              ai = v0 + j;
            }
        }
        // one partial per 64-column chunk: (max y, sum 2^(y - max), argmax)
        if (vrow && v0 < p.V)
          p.part[(size_t)b * p.nparts + v0 / CW] =
              make_float4(mc, (sm[0] + sm[1]) + (sm[2] + sm[3]), av, __int_as_float(ai));
      } else {
        // numerators w = 2^(y - m) (sampled rows), then the draw: the row's
        // select kernel named the chunk where the prefix sum of w crosses u S
        // and the sum before it; the thread walks that chunk in token order
        // with exactly the values it writes.  Rounding that leaves no crossing
        // picks the chunk's last token with positive weight.
        if (sampled) {
#pragma unroll
          for (int j = 0; j < 64; ++j) acc[j] = (j < nvalid) ? exp_shifted(scale_logit(acc[j], c), rm) : 0.f;
        }
        if (v0 / CW == cstar) {
          float run = sbase, pf = 0.f, pl = 0.f;
          int xf = -1, xl = -1;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float wj = acc[j];
            if (wj > 0.f) {
              xl = v0 + j;
              pl = wj;
            }
            run += wj;
            if (xf < 0 && shit && run > starget) {
              xf = v0 + j;
              pf = wj;
            }
          }
          if (xf < 0) {
            xf = xl;
            pf = pl;
          }
          if (xf >= 0) {
            p.tokens[(size_t)b * p.G + p.k] = xf;
            pdtok = __fmul_rn(pf, rinvS);
            have_pdtok = true;
          }
        }
        const int row0 = row_base + q * 32;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // the previous TMA store must have read the staging buffer
          if (lane == 0) ptx::bulk_wait_read0();
          __syncwarp();
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 32 * h + 4 * cc + e;
              const float pr = sampled ? __fmul_rn(acc[j], rinvS) : ((v0 + j == xb) ? 1.f : 0.f);
              if (v0 + j == xb) {
                pdtok = pr;
                have_pdtok = true;
              }
              pv[e] = pr;
            }
            *reinterpret_cast<float4*>(stg + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                make_float4(pv[0], pv[1], pv[2], pv[3]);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.B && v0 + 32 * h < p.V) {  // boxes that start past B or V would write nothing
            // p_d is streamed out: evict-first keeps the re-read W2 in L2
            ptx::tma_store_3d(&tmPd, stg, v0 + 32 * h, p.k, row0, ptx::policy_evict_first());
            ptx::bulk_commit();
          }
        }
      }
    }
    if (WRITE) {
      if (vrow && have_pdtok) p.pd_tok[(size_t)b * p.G + p.k] = pdtok;
      if (lane == 0) ptx::bulk_wait0();
    }
  }

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
  int l2_bytes = 0;
  bool sm103 = false;
};

static DevInfo dev_info() {
  static DevInfo cache[64];
  static bool have[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DevInfo{};
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&cache[dev].l2_bytes, cudaDevAttrL2CacheSize, dev);
    cache[dev].sms = sms;
    cache[dev].sm103 = (major == 10 && minor == 3);
    have[dev] = true;
  }
  return cache[dev];
}

}  // namespace tc

// Which logits path the draft sampler uses: tensor cores when the shape fits
// the tile (bf16, r a multiple of 64 up to 256, V a multiple of 8) on an
// sm_103 device; otherwise the CUDA-core path.  DSPARK_DRAFT_PATH=cuda_core
// forces the CUDA-core path (used by the tests to cover both paths).
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

// vocabulary columns summarised by one partial of the tensor-core pass 1
int draft_tc_tile_width() { return tc::CW; }

cudaError_t draft_tc_prepare(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, TcMaps* maps) {
  const dspark_dims& d = a.dims;
  const cuuint64_t V = (cuuint64_t)d.V, G = (cuuint64_t)d.gamma, B = (cuuint64_t)d.B, r = (cuuint64_t)d.r;
  {  // U [B, G, V] bf16 as (v, k, b)
    const cuuint64_t dims[3] = {V, G, B};
    const cuuint64_t strides[2] = {V * 2, G * V * 2};
    const cuuint32_t box[3] = {tc::CW, 1, tc::BM};
    if (!tc::encode(&maps->U, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.U, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  {  // W2 [r, V] bf16 as (v, i)
    const cuuint64_t dims[2] = {V, r};
    const cuuint64_t strides[1] = {V * 2};
    const cuuint32_t box[2] = {tc::CW, tc::KC};
    if (!tc::encode(&maps->W2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  {  // p_d rows [B, G, V] fp32 as (v, k, b); stores of 32 columns x 32 rows
    const cuuint64_t dims[3] = {V, G, B};
    const cuuint64_t strides[2] = {V * 4, G * V * 4};
    const cuuint32_t box[3] = {32, 1, 32};
    if (!tc::encode(&maps->Pd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.pd_rows, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(tc::k_logits_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)tc::smem_bytes(false));
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(tc::k_logits_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)tc::smem_bytes(true));
  });
  return attr_err;
}

// M-tiles per slab.  The passes of one position run slab by slab (pass 1,
// select, pass 2 of the slab's rows, then the next slab) when a slab's U rows
// and all of W2 fit in about a third of L2: pass 2 then finds both there and
// reads HBM only for the p_d rows it writes.  (On GB300 a buffer read again
// after one pass is found in L2 only up to about 48 MB, and not at all once a
// stream of p_d writes has passed through, whatever the eviction hints.)
// Otherwise a single slab covers the whole batch.  DSPARK_TC_SLAB=<n> forces
// n M-tiles per slab.
int draft_tc_slab_mtiles(const dspark_dims& d) {
  static int forced = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* e = getenv("DSPARK_TC_SLAB");
    forced = e ? atoi(e) : -1;
  });
  const int n_mtiles = (d.B + tc::BM - 1) / tc::BM;
  if (forced > 0) return min(forced, n_mtiles);
  const double w2 = 2.0 * d.r * d.V, u_tile = 2.0 * tc::BM * d.V;
  const double budget = 0.35 * (double)tc::dev_info().l2_bytes;
  const int fit = (int)((budget - w2) / u_tile);
  return fit >= 1 ? min(fit, n_mtiles) : n_mtiles;
}

cudaError_t launch_draft_tc_pass(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, const TcMaps& maps,
                                 int k, bool write, int m_first, int m_count, bool u_keep, cudaStream_t s) {
  const dspark_dims& d = a.dims;
  tc::Params p;
  p.B = d.B;
  p.G = d.gamma;
  p.V = d.V;
  p.r = d.r;
  p.H = d.H;
  p.k = k;
  p.ntiles = (d.V + tc::BN - 1) / tc::BN;
  p.nparts = (d.V + tc::CW - 1) / tc::CW;
  const int sms = tc::dev_info().sms > 0 ? tc::dev_info().sms : 148;
  p.ctas_per_m = max(1, min(p.ntiles, sms / m_count));
  p.m_first = m_first;
  p.u_keep = u_keep ? 1 : 0;
  p.W1 = static_cast<const __nv_bfloat16*>(a.W1);
  p.w = static_cast<const __nv_bfloat16*>(a.w);
  p.zh = reinterpret_cast<const float*>(ws + L.zh);
  p.anchor = a.anchor;
  p.temp = a.temp;
  p.rowstat = reinterpret_cast<const float2*>(ws + L.rowstat);
  p.sel = reinterpret_cast<const float4*>(ws + L.sel);
  p.tokens = a.tokens;
  p.part = reinterpret_cast<float4*>(ws + L.part);
  p.pd_tok = a.pd_tok;
  p.conf_logit = a.conf_logit;
  p.conf = a.conf;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  const dim3 grid(m_count * p.ctas_per_m);
  const size_t smem = tc::smem_bytes(write);
  if (write)
    tc::k_logits_tc<true><<<grid, tc::kThreads, smem, s>>>(maps.U, maps.W2, maps.Pd, p);
  else
    tc::k_logits_tc<false><<<grid, tc::kThreads, smem, s>>>(maps.U, maps.W2, maps.Pd, p);
  return cudaGetLastError();
}

}  // namespace dspark
