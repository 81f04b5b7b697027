// Host-side internals shared by the dspark translation units.
#pragma once

#include <functional>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// Vocabulary columns summarised by one (max, sum-exp, argmax) partial of the
// draft sampler.  The CUDA-core path uses 256, the tensor-core path 64; the
// workspace is sized for the smaller width.
constexpr int kPartialTileMin = 64;

// Slices per kept row in the verify row statistics.
constexpr int RS_PARTS = 4;

// Most vocabulary segments (CTAs per M-tile) of the tensor-core draft kernel.
constexpr int kDraftMaxSeg = 160;

struct WsLayout {
  size_t zh = 0;       // [B*G] f32: w_h . h_k
  size_t E = 0;        // [2][B*r] (f32-sized): the rows the bias product uses, W1 rows (dtype) or RNN rows (f32)
  size_t part = 0;     // [B*ntiles] float4: (tile max, tile sum-exp, argmax value, argmax index);
                       // the fused kernel keeps float2 partials of 64-column chunks there
  size_t rowstat = 0;  // [B] float2: (row max, row sum) of the current position
  size_t sel = 0;      // [B] float4: crossing chunk, prefix before it, target, hit (tensor-core path)
  size_t segpart = 0;  // [B*kDraftMaxSeg] float4: per vocabulary segment partials (tensor-core path)
  size_t gbar = 0;     // u32 grid-barrier counter of the persistent draft kernels, then
                       // [(G+1) * ceil(B/128)] u32 tile counters (16 bytes in)
  size_t sk0 = 0, sk1 = 0, sv0 = 0, sv1 = 0;  // scheduler sort buffers [B*G] u32
  size_t vrs = 0;      // [B*(G+1)*RS_PARTS] float4: verify row-slice statistics
  size_t vm = 0;       // [B] i32: verify accepted count
  size_t vrowT = 0;    // [B*(G+1)] f32: temperature of each kept verify row
  size_t vfmeta = 0;   // [B] int4: final row, rejecting?, sampled?, accepted count
  size_t vfstat = 0;   // [B] float4: final row's max, 1/sum, scale
  size_t vfin = 0;     // [B * 32 ceil(ceil(V/256)/32)] float2: verify chunk sums of the final draw
  size_t rnn_s = 0;    // [2][B*r] f32: RNN head state, positions alternate
  size_t rnn_p = 0;    // [B*gamma][3r] f32: RNN head projections of h
  size_t rnn_z = 0;    // [B][4r] bf16: RNN head z'' of the tensor-core recurrent step
  size_t rnn_wz = 0;   // [3r][4r] bf16: RNN head weights of that step
  size_t rnn_pre = 0;  // [B][3r] f32: its products
  size_t total = 0;
};

WsLayout ws_layout(const dspark_dims& d);

// host-side launch accounting (dspark_launch_count)
void count_launches(int n);

// DSPARK_OK for cudaSuccess; otherwise records e for dspark_last_cuda_error on
// this thread and returns DSPARK_CUDA_ERROR.
dspark_status cuda_status(cudaError_t e);

// The argument checks of the scheduler entry points (dspark_schedule and
// dspark_schedule_noalloc), before anything is enqueued: DSPARK_INVALID_ARG
// for a null or malformed argument, DSPARK_UNSUPPORTED for B * gamma above
// max_keys or an asynchronous batch beyond one CTA's shared memory.  B == 0
// passes (the callers return at once).
dspark_status check_sched_args(const dspark_sched_args* a, int64_t max_keys);

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute belongs to the kernel's instance in each
// device's context, so it is recorded per (device, kernel); a process that
// drives several GPUs gets it set on each.  Thread-safe.
cudaError_t ensure_smem_limit(const void* func, int bytes);
size_t elem_size(int dtype);

// A scheduler run beside the draft kernel's last sweep (dspark_draft_and_schedule).
// want: the caller will launch it behind the draft; on return armed says that
// the fused-sweep kernel ran with a donor CTA and publishes its selects in
// *sel_done, which reaches n_ctas once every confidence and token is written.
struct DraftOverlap {
  bool want = false;
  bool armed = false;
  unsigned* sel_done = nullptr;
  unsigned n_ctas = 0;
};

// Launchers (argument checking happens in capi.cu before these are called).
cudaError_t launch_draft(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s,
                         DraftOverlap* ov = nullptr);
cudaError_t launch_schedule(const dspark_sched_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s);
// whether the asynchronous top-K mode can run at this size (one CTA's shared memory)
bool schedule_async_supported(int B, int G);
// whether the schedule can run behind the draft kernel as one CTA that also
// calibrates the keys: the shared-memory kernel up to 8192 slots, the radix
// kernel above (every size dspark_schedule accepts)
bool schedule_behind_draft_supported(int B, int G);
// that launch with programmatic stream serialization behind the draft kernel,
// waiting for *dep >= dep_target; cudaErrorNotSupported when
// !schedule_behind_draft_supported
cudaError_t launch_schedule_behind_draft(const dspark_sched_args& a, uint8_t* ws, const WsLayout& L,
                                         const unsigned* dep, unsigned dep_target, cudaStream_t s);
cudaError_t launch_verify(const dspark_verify_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s);

// RNN head (rnn_head.cu): P [B gamma, 3r] = the h_j part of every position's
// projection (once per draft call), then the recurrent step of position j
// (1-based): s_j and the fp32 row e_j from s_{j-1} (ignored for j = 1),
// x_{j-1} and P.
cudaError_t launch_rnn_hproj(const dspark_draft_args& a, float* P, WsHeader* hdr, cudaStream_t s);
// the same product on the tensor cores (draft_tc.cu): bf16, H and r multiples of 8
bool rnn_hproj_tc_supported(const dspark_dims& d);
cudaError_t launch_rnn_hproj_tc(const dspark_draft_args& a, float* P, WsHeader* hdr, cudaStream_t s);
// C[M, N] (fp32) = A[M, K] . B[N, K]^T, bf16 operands with K contiguous (draft_tc.cu)
cudaError_t launch_tc_gemm_nt(const void* A, int lda, const void* Bm, int ldb, float* C, int M, int N, int K,
                              WsHeader* hdr, cudaStream_t s);
// the RNN head's recurrent step on the tensor cores (rnn_head.cu): Wz packed
// once per draft call, then per position z'' = [s split in three bf16 parts;
// W1[x]], the GEMM into pre, and the gates
cudaError_t launch_rnn_pack_wz(const dspark_draft_args& a, __nv_bfloat16* Wz, cudaStream_t s);
cudaError_t launch_rnn_step_tc(const dspark_draft_args& a, int j, const float* P, const float* s_prev, float* s_new,
                               __nv_bfloat16* E, __nv_bfloat16* Z, const __nv_bfloat16* Wz, float* pre,
                               WsHeader* hdr, cudaStream_t s);
// (E: [B, r] rows in dims.dtype)
cudaError_t launch_rnn_step(const dspark_draft_args& a, int j, const float* P, const float* s_prev, float* s_new,
                            void* E, cudaStream_t s);

// Verify-batch packing (pack.cu).
cudaError_t launch_pack_rows(const dspark_pack_args& a, WsHeader* hdr, cudaStream_t s);

// STS fitting (sts_fit.cu): its own workspace, after a WsHeader.
struct StsLayout {
  size_t hp = 0;         // [gamma * n_bins * n_grid] u64 fixed-point prediction sums
  size_t hy = 0;         // [gamma * n_bins * n_grid] u32 accepted-prefix counts
  size_t table_end = 0;  // end of the two tables (zeroed per call)
  size_t P = 0;          // [gamma * N] f32 calibrated running products
  size_t gidx = 0;       // [gamma] i32 chosen candidates
  size_t total = 0;
};
StsLayout sts_layout(int N, int G, int n_grid, int n_bins);
cudaError_t launch_sts_fit(const dspark_sts_fit_args& a, uint8_t* ws, const StsLayout& L, cudaStream_t s);

// Tensor-core draft sampler (draft_tc.cu).
bool draft_tc_supported(const dspark_dims& d);
// With a hook, one launch per pass and hook(k) before each position k, whose
// rows the kernel then reads from Erows [B, r] instead of gathering W1 rows
// (the hook also forms the confidences).
cudaError_t launch_draft_tc(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s,
                            const std::function<cudaError_t(int)>* hook = nullptr,
                            const void* Erows = nullptr);
// Fused-sweep kernel (draft_fused.cu); cudaErrorNotSupported when it cannot run.
cudaError_t launch_draft_fused(const dspark_draft_args& a, uint8_t* ws, const WsLayout& L, cudaStream_t s,
                               DraftOverlap* ov = nullptr);

}  // namespace dspark
