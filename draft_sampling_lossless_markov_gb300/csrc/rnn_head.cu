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
// together, so the gate arithmetic needs no second pass.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {

namespace {

constexpr int RN_BM = 16;  // requests per CTA
constexpr int RN_BN = 32;  // state columns per CTA
constexpr int RN_KC = 32;  // z entries per shared-memory chunk
constexpr int RN_THREADS = 256;

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

template <typename T>
__global__ void __launch_bounds__(RN_THREADS) k_rnn_step(const T* __restrict__ Wr, const T* __restrict__ W1,
                                                         const float* __restrict__ P,
                                                         const int32_t* __restrict__ anchor,
                                                         const int32_t* __restrict__ tokens,
                                                         const float* __restrict__ s_prev, float* __restrict__ s_new,
                                                         T* __restrict__ E, int B, int G, int V, int r, int H,
                                                         int j) {
  constexpr int ZPT = RN_BM * RN_KC / RN_THREADS;      // z entries each thread stages per chunk
  constexpr int WPT = 3 * RN_BN * RN_KC / RN_THREADS;  // W entries each thread stages per chunk
  __shared__ float zs[RN_BM][RN_KC + 1];
  __shared__ float ws[3][RN_BN][RN_KC + 1];
  __shared__ int xs[RN_BM];
  const int K = 2 * r, ldw = 2 * r + H;  // the h_j part comes from P
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int c0 = blockIdx.x * RN_BN, b0 = blockIdx.y * RN_BM;
  if (tid < RN_BM) {
    const int b = b0 + tid;
    int x = 0;
    if (b < B) x = (j == 1) ? anchor[b] : tokens[(size_t)b * G + j - 2];
    xs[tid] = (x >= 0 && x < V) ? x : 0;  // out-of-range anchors are reported by the confidence kernel
  }
  __syncthreads();
  // the next chunk's entries are loaded into registers while the current one is used
  float zr[ZPT], wr[WPT];
  auto fetch = [&](int i0) {
#pragma unroll
    for (int u = 0; u < ZPT; ++u) {
      const int idx = tid + u * RN_THREADS;
      const int m = idx / RN_KC, kk = idx - m * RN_KC;
      const int b = b0 + m, i = i0 + kk;
      float v = 0.f;
      if (b < B && i < K) v = (i < r) ? ((j == 1) ? 0.f : s_prev[(size_t)b * r + i])
                                       : to_f32(W1[(size_t)xs[m] * r + (i - r)]);
      zr[u] = v;
    }
#pragma unroll
    for (int u = 0; u < WPT; ++u) {
      const int idx = tid + u * RN_THREADS;
      const int g = idx / (RN_BN * RN_KC);
      const int rem = idx - g * RN_BN * RN_KC;
      const int c = rem / RN_KC, kk = rem - c * RN_KC;
      const int col = c0 + c, i = i0 + kk;
      wr[u] = (col < r && i < K) ? to_f32(Wr[((size_t)g * r + col) * ldw + i]) : 0.f;
    }
  };
  fetch(0);
  float ag[2] = {0.f, 0.f}, ac[2] = {0.f, 0.f}, ao[2] = {0.f, 0.f};
  for (int i0 = 0; i0 < K; i0 += RN_KC) {
    __syncthreads();  // the previous chunk is consumed
#pragma unroll
    for (int u = 0; u < ZPT; ++u) {
      const int idx = tid + u * RN_THREADS;
      zs[idx / RN_KC][idx % RN_KC] = zr[u];
    }
#pragma unroll
    for (int u = 0; u < WPT; ++u) {
      const int idx = tid + u * RN_THREADS;
      const int g = idx / (RN_BN * RN_KC);
      const int rem = idx - g * RN_BN * RN_KC;
      ws[g][rem / RN_KC][rem % RN_KC] = wr[u];
    }
    __syncthreads();
    if (i0 + RN_KC < K) fetch(i0 + RN_KC);
#pragma unroll 8
    for (int kk = 0; kk < RN_KC; ++kk) {
      const float wg = ws[0][tx][kk], wc = ws[1][tx][kk], wo = ws[2][tx][kk];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float z = zs[ty + 8 * q][kk];
        ag[q] = fmaf(wg, z, ag[q]);
        ac[q] = fmaf(wc, z, ac[q]);
        ao[q] = fmaf(wo, z, ao[q]);
      }
    }
  }
  const int col = c0 + tx;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int b = b0 + ty + 8 * q;
    if (b >= B || col >= r) continue;
    float pg = ag[q], pc = ac[q], po = ao[q];
    if (H > 0) {
      const float* pr = P + ((size_t)b * G + (j - 1)) * 3 * r;
      pg += pr[col];
      pc += pr[r + col];
      po += pr[2 * r + col];
    }
    const float g = 1.f / (1.f + expf(-pg));
    const float sp = (j == 1) ? 0.f : s_prev[(size_t)b * r + col];
    s_new[(size_t)b * r + col] = g * sp + (1.f - g) * tanhf(pc);
    store_row(E + (size_t)b * r + col, tanhf(po));
  }
}

}  // namespace

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
  if (d.dtype == DSPARK_BF16)
    k_rnn_step<__nv_bfloat16><<<grid, RN_THREADS, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.W_rnn), static_cast<const __nv_bfloat16*>(a.W1), P, a.anchor, a.tokens,
        s_prev, s_new, static_cast<__nv_bfloat16*>(E), d.B, d.gamma, d.V, d.r, d.H, j);
  else
    k_rnn_step<float><<<grid, RN_THREADS, 0, s>>>(static_cast<const float*>(a.W_rnn), static_cast<const float*>(a.W1),
                                                  P, a.anchor, a.tokens, s_prev, s_new, static_cast<float*>(E), d.B,
                                                  d.gamma, d.V, d.r, d.H, j);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dspark
