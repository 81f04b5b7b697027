// RNN sequential head: the recurrent step of one draft position.
//
// [DSpark] 方法细节, "RNN头的实现": with z_j = [s_{j-1}; W1[x_{j-1}]; h_j] in
// R^{2r+H} and one linear map whose rows split into gate, candidate and output
// parts (W_rnn = [W_g; W_c; W_o], [3r, 2r+H]),
//     g   = sigmoid(W_g z_j),  s_j = g * s_{j-1} + (1 - g) * tanh(W_c z_j),
//     e_j = tanh(W_o z_j),     the row that multiplies W2 in the bias of position j;
// s_0 = 0 and x_0 is the anchor.  e_j is stored in the dtype of W2 (the bias
// product's operand precision, as the Markov head's W1 rows are), rounded to
// nearest-even from fp32; s_j stays fp32.
//
// The h_j part of z does not depend on the recurrence, so one GEMM per draft
// call forms P[b, j, :] = W_rnn[:, 2r:] . h_j for every position:
// [B gamma x H] . [H x 3r], on the tensor cores for bf16 (k_rnn_hproj_tc in
// draft_tc.cu), else here (k_rnn_hproj: 64 x 64 tiles, 4 x 4 outputs per thread).  Each
// position then takes one launch (k_rnn_step): a tiled fp32 GEMM
// [B x 2r] . [2r x 3r] over z' = [s_{j-1}; W1[x_{j-1}]], plus P, whose epilogue
// applies the gates.  A CTA of k_rnn_step holds 16 requests x 32 state columns
// and accumulates the three rows of each column (gate, candidate, output)
// together, so the gate arithmetic needs no second pass; each thread keeps
// 4 requests x 2 columns x 3 rows in registers.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {

namespace {

constexpr int RN_BM = 16;     // requests per CTA
constexpr int RN_BN = 32;     // state columns per CTA
constexpr int RN_KC = 16;     // z entries per shared-memory chunk
constexpr int RN_KG = 4;      // groups of 64 threads, each summing a quarter of z
constexpr int RN_THREADS = 64 * RN_KG;

constexpr int HP_TM = 64, HP_TN = 64, HP_TK = 16;  // k_rnn_hproj tile

// P[m, q] = sum_i h[m, i] W_rnn[q, 2r + i]  (m = b gamma + j - 1, q < 3r)
template <typename T>
__global__ void __launch_bounds__(256) k_rnn_hproj(const T* __restrict__ Wr, const T* __restrict__ h,
                                                   float* __restrict__ P, int M, int N, int H, int ldw, int woff) {
  __shared__ __align__(16) float As[2][HP_TK][HP_TM];  // h tile, k-major
  __shared__ __align__(16) float Bs[2][HP_TK][HP_TN];  // W tile, k-major
  const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;
  const int m0 = blockIdx.y * HP_TM, n0 = blockIdx.x * HP_TN;
  float acc[4][4] = {};
  // each thread loads 4 elements of each tile per chunk: row tid / 4, k (tid % 4) * 4 .. + 3
  const int lr = tid >> 2, lk = (tid & 3) * 4;
  auto load = [&](int buf, int k0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = k0 + lk + e;
      const int m = m0 + lr, n = n0 + lr;
      As[buf][lk + e][lr] = (m < M && k < H) ? to_f32(h[(size_t)m * H + k]) : 0.f;
      Bs[buf][lk + e][lr] = (n < N && k < H) ? to_f32(Wr[(size_t)n * ldw + woff + k]) : 0.f;
    }
  };
  load(0, 0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < H; k0 += HP_TK) {
    if (k0 + HP_TK < H) load(buf ^ 1, k0 + HP_TK);
#pragma unroll
    for (int kk = 0; kk < HP_TK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[buf][kk][tr * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][kk][tc * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    __syncthreads();
    buf ^= 1;
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int m = m0 + tr * 4 + u;
    if (m >= M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int n = n0 + tc * 4 + v;
      if (n < N) P[(size_t)m * N + n] = acc[u][v];
    }
  }
}

__device__ __forceinline__ void store_row(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_row(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// One CTA: RN_BM requests x RN_BN state columns, four groups of 64 threads
// each summing a contiguous quarter of the z entries.  Thread (ty, tx) of a
// group accumulates requests 4 ty .. 4 ty + 3 x columns 2 tx, 2 tx + 1 x the
// three rows of each column (gate, candidate, output): 24 fma chains over its
// quarter in ascending order; the quarters are then added in order.  z and
// the weight rows go through shared memory k-major, RN_KC entries at a time;
// the next chunk's global loads are in flight while the current one is used.
// kVec: vector loads (bf16 weights and W1 rows, r % RN_KC == 0, 2r + H % 8 == 0).
template <typename T, bool kVec>
__global__ void __launch_bounds__(RN_THREADS) k_rnn_step(const T* __restrict__ Wr, const T* __restrict__ W1,
                                                         const float* __restrict__ P,
                                                         const int32_t* __restrict__ anchor,
                                                         const int32_t* __restrict__ tokens,
                                                         const float* __restrict__ s_prev, float* __restrict__ s_new,
                                                         T* __restrict__ E, int B, int G, int V, int r, int H,
                                                         int j) {
  // staging (z and weights per group), reused for the groups' sums after the loop
  constexpr int kZs = RN_KG * RN_KC * RN_BM, kWs = RN_KG * 3 * RN_KC * RN_BN, kRed = (RN_KG - 1) * 3 * RN_BM * RN_BN;
  static_assert(kRed <= kZs + kWs, "reduction buffer");
  __shared__ __align__(16) float smem[kZs + kWs];
  __shared__ int xs[RN_BM];
  auto zs = reinterpret_cast<float(*)[RN_KC][RN_BM]>(smem);
  auto ws = reinterpret_cast<float(*)[3][RN_KC][RN_BN]>(smem + kZs);
  auto red = reinterpret_cast<float(*)[3][RN_BM][RN_BN]>(smem);
  const int K = 2 * r, ldw = 2 * r + H;  // the h_j part comes from P
  const int kg = threadIdx.x >> 6, tid = threadIdx.x & 63;
  const int ty = tid >> 4, tx = tid & 15;
  const int c0 = blockIdx.x * RN_BN, b0 = blockIdx.y * RN_BM;
  if (threadIdx.x < RN_BM) {
    const int b = b0 + threadIdx.x;
    int x = 0;
    if (b < B) x = (j == 1) ? anchor[b] : tokens[(size_t)b * G + j - 2];
    xs[threadIdx.x] = (x >= 0 && x < V) ? x : 0;  // out-of-range anchors are reported by the confidence kernel
  }
  __syncthreads();
  // this group's quarter of the z entries, in whole chunks
  const int nch = (K + RN_KC - 1) / RN_KC;
  const int per = (nch + RN_KG - 1) / RN_KG;
  const int ch0 = kg * per, ch1 = min(nch, ch0 + per);
  // staging: thread tid loads z entries kz .. kz + 3 of request mz, and entries
  // kw .. kw + 7 of the three weight rows of column cw
  const int mz = tid >> 2, kz = (tid & 3) * 4;
  const int cw = tid >> 1, kw = (tid & 1) * 8;
  float zr[4], wr[3][8];
  auto fetch = [&](int i0) {
    const int b = b0 + mz;
    const int col = c0 + cw;
    if constexpr (kVec) {
      // a chunk lies wholly in the state part or wholly in the W1 part
      if (b < B && i0 + kz < K) {
        if (i0 < r) {
          if (j == 1) {
#pragma unroll
            for (int u = 0; u < 4; ++u) zr[u] = 0.f;
          } else {
            const float4 s0 = *reinterpret_cast<const float4*>(s_prev + (size_t)b * r + i0 + kz);
            zr[0] = s0.x;
            zr[1] = s0.y;
            zr[2] = s0.z;
            zr[3] = s0.w;
          }
        } else {
          const uint2 q = *reinterpret_cast<const uint2*>(W1 + (size_t)xs[mz] * r + (i0 - r) + kz);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float2 f = __bfloat1622float2(h2[u]);
            zr[2 * u] = f.x;
            zr[2 * u + 1] = f.y;
          }
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) zr[u] = 0.f;
      }
#pragma unroll
      for (int g = 0; g < 3; ++g) {
        if (col < r && i0 + kw < K) {
          const uint4 q = *reinterpret_cast<const uint4*>(Wr + ((size_t)g * r + col) * ldw + i0 + kw);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 f = __bfloat1622float2(h2[u]);
            wr[g][2 * u] = f.x;
            wr[g][2 * u + 1] = f.y;
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) wr[g][u] = 0.f;
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + kz + u;
        float v = 0.f;
        if (b < B && i < K) v = (i < r) ? ((j == 1) ? 0.f : s_prev[(size_t)b * r + i])
                                         : to_f32(W1[(size_t)xs[mz] * r + (i - r)]);
        zr[u] = v;
      }
#pragma unroll
      for (int g = 0; g < 3; ++g)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + kw + u;
          wr[g][u] = (col < r && i < K) ? to_f32(Wr[((size_t)g * r + col) * ldw + i]) : 0.f;
        }
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int u = 0; u < 4; ++u) zs[kg][kz + u][mz] = zr[u];
#pragma unroll
    for (int g = 0; g < 3; ++g)
#pragma unroll
      for (int u = 0; u < 8; ++u) ws[kg][g][kw + u][cw] = wr[g][u];
  };
  float acc[3][4][2];
#pragma unroll
  for (int g = 0; g < 3; ++g)
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[g][u][0] = acc[g][u][1] = 0.f;
  // every group runs the same number of rounds, so that the CTA barriers match
  if (ch0 < ch1) fetch(ch0 * RN_KC);
  for (int c = 0; c < per; ++c) {
    const int ch = ch0 + c;
    const bool live = ch < ch1;
    if (live) stash();
    __syncthreads();
    if (live && ch + 1 < ch1) fetch((ch + 1) * RN_KC);
    if (live) {
#pragma unroll 8
      for (int kk = 0; kk < RN_KC; ++kk) {
        const float4 z4 = *reinterpret_cast<const float4*>(&zs[kg][kk][4 * ty]);
        const float zv[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
        for (int g = 0; g < 3; ++g) {
          const float2 w2 = *reinterpret_cast<const float2*>(&ws[kg][g][kk][2 * tx]);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[g][u][0] = fmaf(w2.x, zv[u], acc[g][u][0]);
            acc[g][u][1] = fmaf(w2.y, zv[u], acc[g][u][1]);
          }
        }
      }
    }
    __syncthreads();
  }
  // groups 1..3 hand their sums to group 0, which adds them in group order
  // (the staging area is free: the loop ended with a barrier)
  if (kg > 0) {
#pragma unroll
    for (int g = 0; g < 3; ++g)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        red[kg - 1][g][4 * ty + u][2 * tx] = acc[g][u][0];
        red[kg - 1][g][4 * ty + u][2 * tx + 1] = acc[g][u][1];
      }
  }
  __syncthreads();
  if (kg > 0) return;
#pragma unroll
  for (int q = 0; q < RN_KG - 1; ++q)
#pragma unroll
    for (int g = 0; g < 3; ++g)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[g][u][0] = __fadd_rn(acc[g][u][0], red[q][g][4 * ty + u][2 * tx]);
        acc[g][u][1] = __fadd_rn(acc[g][u][1], red[q][g][4 * ty + u][2 * tx + 1]);
      }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int b = b0 + 4 * ty + u;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int col = c0 + 2 * tx + v;
      if (b >= B || col >= r) continue;
      float pg = acc[0][u][v], pc = acc[1][u][v], po = acc[2][u][v];
      if (H > 0) {
        const float* pr = P + ((size_t)b * G + (j - 1)) * 3 * r;
        pg += pr[col];
        pc += pr[r + col];
        po += pr[2 * r + col];
      }
      const float gt = 1.f / (1.f + expf(-pg));
      const float sp = (j == 1) ? 0.f : s_prev[(size_t)b * r + col];
      s_new[(size_t)b * r + col] = gt * sp + (1.f - gt) * tanhf(pc);
      store_row(E + (size_t)b * r + col, tanhf(po));
    }
  }
}

// ---- the recurrent step on the tensor cores (bf16, sm_103a) ----
// pre = W_rnn[:, :2r] . z' as one bf16 GEMM with fp32 accumulation.  s_{j-1}
// (fp32) is split into three bf16 parts hi + mid + lo, each the nearest bf16 to
// what the parts before it leave (the remainders are exact in fp32), so that
// the parts carry s to about 2^-27 of its magnitude; z'' = [hi; mid; lo;
// W1[x_{j-1}]] in R^{4r} meets Wz = [W_s, W_s, W_s, W_x] (W_s = W_rnn[:, :r],
// W_x = W_rnn[:, r:2r]), [3r, 4r], packed once per draft call.  Products of
// bf16 operands are exact in fp32; the GEMM adds them in fp32, in another
// order than k_rnn_step's fma chains.

// Wz row n (n < 3r): W_s row n three times, then W_x row n
__global__ void k_rnn_pack_wz(const __nv_bfloat16* __restrict__ Wr, __nv_bfloat16* __restrict__ Wz, int r, int ldw) {
  const int n = blockIdx.y;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 4 * r; i += gridDim.x * blockDim.x)
    Wz[(size_t)n * 4 * r + i] = Wr[(size_t)n * ldw + (i < 3 * r ? i % r : i - 2 * r)];
}

// z'' of request b = blockIdx.y for position j (s_0 = 0, x_0 the anchor)
__global__ void k_rnn_zsplit(const float* __restrict__ s_prev, const __nv_bfloat16* __restrict__ W1,
                             const int32_t* __restrict__ anchor, const int32_t* __restrict__ tokens,
                             __nv_bfloat16* __restrict__ Z, int G, int V, int r, int j) {
  const int b = blockIdx.y;
  int x = (j == 1) ? anchor[b] : tokens[(size_t)b * G + j - 2];
  x = (x >= 0 && x < V) ? x : 0;  // out-of-range anchors are reported by the confidence kernel
  __nv_bfloat16* z = Z + (size_t)b * 4 * r;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < r; i += gridDim.x * blockDim.x) {
    const float s = (j == 1) ? 0.f : s_prev[(size_t)b * r + i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(s);
    const float r1 = __fsub_rn(s, __bfloat162float(hi));
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    z[i] = hi;
    z[r + i] = mid;
    z[2 * r + i] = __float2bfloat16_rn(r2);
    z[3 * r + i] = W1[(size_t)x * r + i];
  }
}

// the gates of position j from pre [B, 3r] (and P), as k_rnn_step's epilogue
__global__ void k_rnn_gates(const float* __restrict__ pre, const float* __restrict__ P,
                            const float* __restrict__ s_prev, float* __restrict__ s_new,
                            __nv_bfloat16* __restrict__ E, int B, int G, int r, int H, int j) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * r) return;
  const int b = idx / r, col = idx - b * r;
  const float* pb = pre + (size_t)b * 3 * r;
  float pg = pb[col], pc = pb[r + col], po = pb[2 * r + col];
  if (H > 0) {
    const float* pr = P + ((size_t)b * G + (j - 1)) * 3 * r;
    pg += pr[col];
    pc += pr[r + col];
    po += pr[2 * r + col];
  }
  const float gt = 1.f / (1.f + expf(-pg));
  const float sp = (j == 1) ? 0.f : s_prev[(size_t)b * r + col];
  s_new[(size_t)b * r + col] = gt * sp + (1.f - gt) * tanhf(pc);
  E[(size_t)b * r + col] = __float2bfloat16_rn(tanhf(po));
}

}  // namespace

cudaError_t launch_rnn_pack_wz(const dspark_draft_args& a, __nv_bfloat16* Wz, cudaStream_t s) {
  const dspark_dims& d = a.dims;
  const dim3 grid((4 * d.r + 255) / 256, 3 * d.r);
  k_rnn_pack_wz<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(a.W_rnn), Wz, d.r, 2 * d.r + d.H);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_rnn_step_tc(const dspark_draft_args& a, int j, const float* P, const float* s_prev, float* s_new,
                               __nv_bfloat16* E, __nv_bfloat16* Z, const __nv_bfloat16* Wz, float* pre,
                               WsHeader* hdr, cudaStream_t s) {
  const dspark_dims& d = a.dims;
  const int B = d.B, r = d.r;
  k_rnn_zsplit<<<dim3((r + 255) / 256, B), 256, 0, s>>>(s_prev, static_cast<const __nv_bfloat16*>(a.W1), a.anchor,
                                                         a.tokens, Z, d.gamma, d.V, r, j);
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_tc_gemm_nt(Z, 4 * r, Wz, 4 * r, pre, B, 3 * r, 4 * r, hdr, s);
  if (e != cudaSuccess) return e;
  k_rnn_gates<<<(B * r + 255) / 256, 256, 0, s>>>(pre, P, s_prev, s_new, E, B, d.gamma, r, d.H, j);
  count_launches(1);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_hproj_t(const dspark_draft_args& a, float* P, cudaStream_t s) {
  const dspark_dims& d = a.dims;
  const int M = d.B * d.gamma, N = 3 * d.r;
  const dim3 grid((N + HP_TN - 1) / HP_TN, (M + HP_TM - 1) / HP_TM);
  k_rnn_hproj<T><<<grid, 256, 0, s>>>(static_cast<const T*>(a.W_rnn), static_cast<const T*>(a.h), P, M, N, d.H,
                                      2 * d.r + d.H, 2 * d.r);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_rnn_hproj(const dspark_draft_args& a, float* P, WsHeader* hdr, cudaStream_t s) {
  if (a.dims.H == 0 || a.dims.B == 0) return cudaSuccess;
  if (rnn_hproj_tc_supported(a.dims)) return launch_rnn_hproj_tc(a, P, hdr, s);
  if (a.dims.dtype == DSPARK_BF16) return launch_hproj_t<__nv_bfloat16>(a, P, s);
  return launch_hproj_t<float>(a, P, s);
}

cudaError_t launch_rnn_step(const dspark_draft_args& a, int j, const float* P, const float* s_prev, float* s_new,
                            void* E, cudaStream_t s) {
  const dspark_dims& d = a.dims;
  const dim3 grid((d.r + RN_BN - 1) / RN_BN, (d.B + RN_BM - 1) / RN_BM);
  // vector loads when every chunk lies in one part of z and the rows are 16-byte aligned
  const bool vec = d.dtype == DSPARK_BF16 && d.r % RN_KC == 0 && (2 * d.r + d.H) % 8 == 0 &&
                   (reinterpret_cast<uintptr_t>(a.W_rnn) % 16) == 0 && (reinterpret_cast<uintptr_t>(a.W1) % 16) == 0 &&
                   (reinterpret_cast<uintptr_t>(s_prev) % 16) == 0;
  if (d.dtype == DSPARK_BF16) {
    const auto* Wr = static_cast<const __nv_bfloat16*>(a.W_rnn);
    const auto* W1 = static_cast<const __nv_bfloat16*>(a.W1);
    auto* Eo = static_cast<__nv_bfloat16*>(E);
    if (vec)
      k_rnn_step<__nv_bfloat16, true><<<grid, RN_THREADS, 0, s>>>(Wr, W1, P, a.anchor, a.tokens, s_prev, s_new, Eo,
                                                                 d.B, d.gamma, d.V, d.r, d.H, j);
    else
      k_rnn_step<__nv_bfloat16, false><<<grid, RN_THREADS, 0, s>>>(Wr, W1, P, a.anchor, a.tokens, s_prev, s_new, Eo,
                                                                  d.B, d.gamma, d.V, d.r, d.H, j);
  } else {
    k_rnn_step<float, false><<<grid, RN_THREADS, 0, s>>>(static_cast<const float*>(a.W_rnn),
                                                         static_cast<const float*>(a.W1), P, a.anchor, a.tokens,
                                                         s_prev, s_new, static_cast<float*>(E), d.B, d.gamma, d.V,
                                                         d.r, d.H, j);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dspark
