// Tensor-core (tcgen05) logits passes of the draft sampler, sm_103a.
//
// The Markov-head bias of position k is a dense contraction
//     bias[b, v] = E[b, :] . W2[:, v],   E[b] = W1[x_{k-1}]      (B x r x V)
// ([DSpark] 方法细节, "马尔可夫头（Markov head）的实现").  With r = 256 it is
// 2 r = 512 flop per (b, v) against 6 bytes of U read + p_d write, i.e. far
// above the CUDA-core ridge, so it runs on the 5th-generation tensor cores:
//
//   tile      128 requests (TMEM lanes) x 64 vocabulary columns, K = r
//   warp 0    TMA producer: W2 tile [r x 64] (L2 evict-last: W2 is re-read at
//             every position) and U tile [128 x 64] (L2 evict-first: streamed),
//             both 128B-swizzled, into an NS-deep ring of stages
//   warp 1    allocates TMEM, issues tcgen05.mma (A = E, K-major, resident for
//             the whole CTA; B = W2 tile, MN-major) into one of two 64-column
//             fp32 accumulators, commits to mbarriers
//   warps 2-9 epilogue, two groups of four warps (one per TMEM lane quarter)
//             that take alternate tiles, each with its own accumulator: one
//             request row per thread, TMEM -> registers, + U, then either the
//             tile's (max, sum, argmax) partial (pass 1) or the probability
//             row p_d = 2^(y - m) / S written through a per-warp swizzled
//             staging buffer with TMA stores (pass 2)
//
// A CTA owns one 128-row M-tile and a contiguous run of vocabulary tiles, so
// its E tile is loaded once.  Every mbarrier wait gives up after two seconds:
// the kernel then records DSPARK_TIMEOUT in the workspace error word, lets the
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

constexpr int BM = 128;
constexpr int BN = 64;
constexpr int kEpiGroups = 2;                       // epilogue groups of 4 warps
constexpr int kThreads = 64 + kEpiGroups * 128;     // producer, MMA, epilogue
constexpr int kEpiWarp0 = 2;
constexpr int kStagingPerWarp = 32 * 64 * 4;        // [32 rows x 64 cols] fp32
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kTmemCols = 128;  // two 64-column accumulators

struct Params {
  int B, G, V, r, k, ntiles, ctas_per_m;
  const float* temp;
  const float2* rowstat;
  const int32_t* tokens;
  float4* part;
  float* pd_tok;
  WsHeader* hdr;
};

__host__ __device__ constexpr int num_stages(bool write) { return write ? 2 : 3; }

__host__ __device__ inline size_t smem_bytes(int r, bool write) {
  const size_t e_bytes = (size_t)r * 256;             // BM rows x r cols bf16
  const size_t stage = (size_t)r * 128 + BM * 128;    // W2 [r x 64] + U [128 x 64], bf16
  const size_t staging = write ? (size_t)kEpiGroups * 4 * kStagingPerWarp : 0;
  return 1024 + e_bytes + num_stages(write) * stage + staging + 256;
}

template <bool WRITE>
__global__ void __launch_bounds__(kThreads, 1)
    k_logits_tc(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmW2,
                const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmPd, Params p) {
  constexpr int NS = num_stages(WRITE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int r = p.r;
  const uint32_t e_bytes = (uint32_t)r * 256;
  const uint32_t w2_bytes = (uint32_t)r * 128;
  const uint32_t stage_bytes = w2_bytes + BM * 128;
  uint8_t* sE = smem;
  uint8_t* sStage = sE + e_bytes;
  uint8_t* sStg = sStage + NS * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + (WRITE ? kEpiGroups * 4 * kStagingPerWarp : 0));
  uint64_t* full = bars;
  uint64_t* empty = bars + NS;
  uint64_t* tfull = bars + 2 * NS;
  uint64_t* tempty = tfull + 2;
  uint64_t* efull = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(efull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x / p.ctas_per_m;
  const int part_i = blockIdx.x % p.ctas_per_m;
  const int n_per = (p.ntiles + p.ctas_per_m - 1) / p.ctas_per_m;
  const int n_lo = min(part_i * n_per, p.ntiles);
  const int count = min(p.ntiles, n_lo + n_per) - n_lo;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1 + 4);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 4);
    }
    ptx::mbar_init(efull, 1);
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
      ptx::mbar_expect_tx(efull, e_bytes);
      for (int kb = 0; kb < r / 64; ++kb)
        ptx::tma_load_2d(sE + kb * (BM * 128), &tmE, efull, kb * 64, m_tile * BM, pol_last);
      int issued = 0;
      for (int i = 0; i < count; ++i) {
        const int s = i % NS;
        if (!ptx::mbar_wait(&empty[s], ((i / NS) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
          fail();
          break;
        }
        const int n = n_lo + i;
        uint8_t* st = sStage + s * stage_bytes;
        ptx::mbar_expect_tx(&full[s], stage_bytes);
        ptx::tma_load_2d(st, &tmW2, &full[s], n * BN, 0, pol_last);
        ptx::tma_load_3d(st + w2_bytes, &tmU, &full[s], n * BN, p.k, m_tile * BM, pol_first);
        issued = i + 1;
      }
      // every load this thread issued has landed before the CTA may exit
      ptx::mbar_wait(efull, 0, abort_flag, kWaitLimitNs);
      for (int i = max(0, issued - NS); i < issued; ++i)
        ptx::mbar_wait(&full[i % NS], (i / NS) & 1, abort_flag, kWaitLimitNs);
    }
  } else if (count > 0 && warp == 1) {
    // ------------------------------ MMA issuer --------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, false, true);
      const uint32_t aE = ptx::smem_u32(sE);
      int issued = 0;
      if (ptx::mbar_wait(efull, 0, abort_flag, kWaitLimitNs)) {
        for (int i = 0; i < count; ++i) {
          const int s = i % NS, a = i & 1;
          if (!ptx::mbar_wait(&full[s], (i / NS) & 1, abort_flag, kWaitLimitNs) ||
              !ptx::mbar_wait(&tempty[a], ((i >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs)) {
            fail();
            break;
          }
          ptx::tc_fence_after();
          const uint32_t aW2 = ptx::smem_u32(sStage + s * stage_bytes);
          const uint32_t d = tmem + (uint32_t)(a * BN);
          for (int ks = 0; ks < r / 16; ++ks) {
            // A: E tile, K-major, 128B swizzle: 64-column blocks of BM x 128 B,
            //    K steps of 16 advance 32 B inside a block; 8-row groups 1024 B apart
            const uint64_t ad = ptx::smem_desc_sw128(aE + (ks >> 2) * (BM * 128) + (ks & 3) * 32, 16, 1024);
            // B: W2 tile [r x 64], MN-major, 128B swizzle: rows of 128 B (64 columns),
            //    8-row groups 1024 B apart along K, a K step of 16 is two groups
            //    (the leading offset only matters for tiles wider than 64 columns)
            const uint64_t bd = ptx::smem_desc_sw128(aW2 + ks * 2048, 16, 1024);
            ptx::tc_mma(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
          }
          ptx::tc_commit(&empty[s]);
          ptx::tc_commit(&tfull[a]);
          issued = i + 1;
        }
      } else {
        fail();
      }
      // the last commit tracks every MMA issued: TMEM is not freed under a running MMA
      if (issued > 0)
        ptx::mbar_wait(&tfull[(issued - 1) & 1], ((issued - 1) >> 1) & 1, abort_flag, kWaitLimitNs);
    }
  } else if (count > 0 && warp >= kEpiWarp0) {
    // ------------------------------ epilogue ----------------------------------
    const int g = (warp - kEpiWarp0) >> 2;  // epilogue group: tiles i with i % 2 == g
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int b = m_tile * BM + row;
    const bool vrow = b < p.B;
    const float T_ = vrow ? p.temp[b] : 1.f;
    const bool sampled = T_ > 0.f;
    const float c = row_scale(T_);
    float rm = 0.f, rinvS = 1.f;
    int xb = -1;
    if (WRITE && vrow) {
      const float2 st = p.rowstat[b];
      rm = st.x;
      rinvS = inv_sum(st.y);
      xb = p.tokens[(size_t)b * p.G + p.k];
    }
    uint8_t* stg = sStg + (warp - kEpiWarp0) * kStagingPerWarp;
    float pdtok = 0.f;
    bool have_pdtok = false;
    for (int i = g; i < count; i += kEpiGroups) {
      const int s = i % NS, a = i & 1;
      const int n = n_lo + i;
      const int v0 = n * BN;
      bool ok = ptx::mbar_wait(&tfull[a], (i >> 1) & 1, abort_flag, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) fail();
        break;
      }
      ptx::tc_fence_after();
      float acc[64];
      {
        float h0[32], h1[32];
        const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN);
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
      ok = ptx::mbar_wait(&full[s], (i / NS) & 1, abort_flag, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) fail();
        break;
      }
      // U row of this thread: 8 swizzled 16-byte chunks of 8 bf16
      const uint8_t* su = sStage + s * stage_bytes + w2_bytes + row * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const uint4 qv = *reinterpret_cast<const uint4*>(su + ((cc ^ (row & 7)) << 4));
        const __nv_bfloat162* bp = reinterpret_cast<const __nv_bfloat162*>(&qv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(bp[e]);
          acc[8 * cc + 2 * e] = add_base(f.x, acc[8 * cc + 2 * e]);
          acc[8 * cc + 2 * e + 1] = add_base(f.y, acc[8 * cc + 2 * e + 1]);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[s]);
      // acc[j] now holds the logit l of column v0 + j; columns past V are masked
      const int nvalid = min(BN, p.V - v0);
      if (!WRITE) {
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          acc[j] = (j < nvalid) ? scale_logit(acc[j], c) : -INFINITY;  // y = l c (greedy rows: c = 1)
          mx[j & 3] = fmaxf(mx[j & 3], acc[j]);
        }
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        float sm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 64; ++j) sm[j & 3] += exp_shifted(acc[j], mt);
        const float st = (sm[0] + sm[1]) + (sm[2] + sm[3]);
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
        if (vrow) p.part[(size_t)b * p.ntiles + n] = make_float4(mt, st, av, __int_as_float(ai));
      } else {
        // the previous tile's TMA stores must have read the staging buffer
        if (lane == 0) ptx::bulk_wait_read0();
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 32 * h + 4 * cc + e;
              const float pr = sampled ? prob_from(scale_logit(acc[j], c), rm, rinvS) : ((v0 + j == xb) ? 1.f : 0.f);
              if (v0 + j == xb) {
                pdtok = pr;
                have_pdtok = true;
              }
              pv[e] = pr;
            }
            *reinterpret_cast<float4*>(stg + h * 4096 + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
                make_float4(pv[0], pv[1], pv[2], pv[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        const int row0 = m_tile * BM + q * 32;
        if (lane == 0 && row0 < p.B) {  // boxes that start past B or V would write nothing
          ptx::tma_store_3d(&tmPd, stg, v0, p.k, row0);
          if (v0 + 32 < p.V) ptx::tma_store_3d(&tmPd, stg + 4096, v0 + 32, p.k, row0);
          ptx::bulk_commit();
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
  if (d.dtype != DSPARK_BF16 || d.r < 64 || d.r > 256 || (d.r % 64) != 0 || (d.V % 8) != 0) return false;
  return tc::dev_info().sm103 && tc::encode_fn() != nullptr;
}

int draft_tc_tile_width() { return tc::BN; }

cudaError_t draft_tc_prepare(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, TcMaps* maps) {
  const dspark_dims& d = a.dims;
  const cuuint64_t V = (cuuint64_t)d.V, G = (cuuint64_t)d.gamma, B = (cuuint64_t)d.B, r = (cuuint64_t)d.r;
  {  // U [B, G, V] bf16 as (v, k, b)
    const cuuint64_t dims[3] = {V, G, B};
    const cuuint64_t strides[2] = {V * 2, G * V * 2};
    const cuuint32_t box[3] = {tc::BN, 1, tc::BM};
    if (!tc::encode(&maps->U, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.U, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  {  // W2 [r, V] bf16 as (v, i)
    const cuuint64_t dims[2] = {V, r};
    const cuuint64_t strides[1] = {V * 2};
    const cuuint32_t box[2] = {tc::BN, (cuuint32_t)r};
    if (!tc::encode(&maps->W2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  for (int eb = 0; eb < 2; ++eb) {  // E [2][B, r] bf16 (workspace) as (i, b), one map per buffer
    const cuuint64_t dims[2] = {r, B};
    const cuuint64_t strides[1] = {r * 2};
    const cuuint32_t box[2] = {64, tc::BM};
    if (!tc::encode(&maps->E[eb], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ws + L.E + (size_t)eb * B * r * 2, dims, strides,
                    box))
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
                                    (int)tc::smem_bytes(256, false));
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(tc::k_logits_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)tc::smem_bytes(256, true));
  });
  return attr_err;
}

cudaError_t launch_draft_tc_pass(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, const TcMaps& maps,
                                 int k, bool write, cudaStream_t s) {
  const dspark_dims& d = a.dims;
  tc::Params p;
  p.B = d.B;
  p.G = d.gamma;
  p.V = d.V;
  p.r = d.r;
  p.k = k;
  p.ntiles = (d.V + tc::BN - 1) / tc::BN;
  const int n_mtiles = (d.B + tc::BM - 1) / tc::BM;
  const int sms = tc::dev_info().sms > 0 ? tc::dev_info().sms : 148;
  p.ctas_per_m = max(1, min(p.ntiles, sms / n_mtiles));
  p.temp = a.temp;
  p.rowstat = reinterpret_cast<const float2*>(ws + L.rowstat);
  p.tokens = a.tokens;
  p.part = reinterpret_cast<float4*>(ws + L.part);
  p.pd_tok = a.pd_tok;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  const dim3 grid(n_mtiles * p.ctas_per_m);
  const size_t smem = tc::smem_bytes(d.r, write);
  if (write)
    tc::k_logits_tc<true><<<grid, tc::kThreads, smem, s>>>(maps.U, maps.W2, maps.E[k & 1], maps.Pd, p);
  else
    tc::k_logits_tc<false><<<grid, tc::kThreads, smem, s>>>(maps.U, maps.W2, maps.E[k & 1], maps.Pd, p);
  return cudaGetLastError();
}

}  // namespace dspark
