// RNN sequential head: the recurrent step of one draft position.
//
// [DSpark] 方法细节, "RNN头的实现": with z_j = [s_{j-1}; W1[x_{j-1}]; h_j] in
// R^{2r+H} and one linear map whose rows split into gate, candidate and output
// parts (W_rnn = [W_g; W_c; W_o], [3r, 2r+H]),
//     g   = sigmoid(W_g z_j),  s_j = g * s_{j-1} + (1 - g) * tanh(W_c z_j),
//     e_j = tanh(W_o z_j),     the row that multiplies W2 in the bias of position j;
// s_0 = 0 and x_0 is the anchor.
//
// One launch per position: a tiled fp32 GEMM [B x (2r+H)] . [(2r+H) x 3r] whose
// epilogue applies the gates.  A CTA holds 16 requests x 32 state columns and
// accumulates the three rows of each column (gate, candidate, output) together,
// so the gate arithmetic needs no second pass.  z is assembled on the fly from
// the state, the embedding row and the hidden state.
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

template <typename T>
__global__ void __launch_bounds__(RN_THREADS) k_rnn_step(const T* __restrict__ Wr, const T* __restrict__ W1,
                                                         const T* __restrict__ h, const int32_t* __restrict__ anchor,
                                                         const int32_t* __restrict__ tokens,
                                                         const float* __restrict__ s_prev, float* __restrict__ s_new,
                                                         float* __restrict__ E, int B, int G, int V, int r, int H,
                                                         int j) {
  __shared__ float zs[RN_BM][RN_KC + 1];
  __shared__ float ws[3][RN_BN][RN_KC + 1];
  __shared__ int xs[RN_BM];
  const int K = 2 * r + H;
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int c0 = blockIdx.x * RN_BN, b0 = blockIdx.y * RN_BM;
  if (tid < RN_BM) {
    const int b = b0 + tid;
    int x = 0;
    if (b < B) x = (j == 1) ? anchor[b] : tokens[(size_t)b * G + j - 2];
    xs[tid] = (x >= 0 && x < V) ? x : 0;  // out-of-range anchors are reported by the confidence kernel
  }
  float ag[2] = {0.f, 0.f}, ac[2] = {0.f, 0.f}, ao[2] = {0.f, 0.f};
  for (int i0 = 0; i0 < K; i0 += RN_KC) {
    __syncthreads();  // the previous chunk is consumed (and xs is written)
    for (int idx = tid; idx < RN_BM * RN_KC; idx += RN_THREADS) {
      const int m = idx / RN_KC, kk = idx - m * RN_KC;
      const int b = b0 + m, i = i0 + kk;
      float v = 0.f;
      if (b < B && i < K) {
        if (i < r)
          v = (j == 1) ? 0.f : s_prev[(size_t)b * r + i];
        else if (i < 2 * r)
          v = to_f32(W1[(size_t)xs[m] * r + (i - r)]);
        else
          v = to_f32(h[((size_t)b * G + (j - 1)) * H + (i - 2 * r)]);
      }
      zs[m][kk] = v;
    }
    for (int idx = tid; idx < 3 * RN_BN * RN_KC; idx += RN_THREADS) {
      const int g = idx / (RN_BN * RN_KC);
      const int rem = idx - g * RN_BN * RN_KC;
      const int c = rem / RN_KC, kk = rem - c * RN_KC;
      const int col = c0 + c, i = i0 + kk;
      ws[g][c][kk] = (col < r && i < K) ? to_f32(Wr[((size_t)g * r + col) * K + i]) : 0.f;
    }
    __syncthreads();
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
    const float g = 1.f / (1.f + expf(-ag[q]));
    const float sp = (j == 1) ? 0.f : s_prev[(size_t)b * r + col];
    s_new[(size_t)b * r + col] = g * sp + (1.f - g) * tanhf(ac[q]);
    E[(size_t)b * r + col] = tanhf(ao[q]);
  }
}

}  // namespace

cudaError_t launch_rnn_step(const dspark_draft_args& a, int j, const float* s_prev, float* s_new, float* E,
                            cudaStream_t s) {
  const dspark_dims& d = a.dims;
  const dim3 grid((d.r + RN_BN - 1) / RN_BN, (d.B + RN_BM - 1) / RN_BM);
  if (d.dtype == DSPARK_BF16)
    k_rnn_step<__nv_bfloat16><<<grid, RN_THREADS, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.W_rnn), static_cast<const __nv_bfloat16*>(a.W1),
        static_cast<const __nv_bfloat16*>(a.h), a.anchor, a.tokens, s_prev, s_new, E, d.B, d.gamma, d.V, d.r, d.H, j);
  else
    k_rnn_step<float><<<grid, RN_THREADS, 0, s>>>(static_cast<const float*>(a.W_rnn), static_cast<const float*>(a.W1),
                                                  static_cast<const float*>(a.h), a.anchor, a.tokens, s_prev, s_new, E,
                                                  d.B, d.gamma, d.V, d.r, d.H, j);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dspark
