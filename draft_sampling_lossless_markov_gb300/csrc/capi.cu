// C ABI of the dspark library: argument checks, workspace layout, dispatch.
// Every check happens before anything is enqueued; nothing here allocates.
#include <algorithm>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "dspark.h"
#include "internal.h"

namespace dspark {

size_t elem_size(int dtype) { return dtype == DSPARK_BF16 ? 2 : 4; }

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static bool dims_ok(const dspark_dims& d) {
  if (d.B < 0 || d.gamma < 1 || d.gamma > DSPARK_MAX_GAMMA || d.V < 1 || d.V > DSPARK_MAX_VOCAB) return false;
  if (d.r < 0 || d.r > DSPARK_MAX_RANK || d.H < 0) return false;
  if (d.dtype != DSPARK_BF16 && d.dtype != DSPARK_F32) return false;
  // index arithmetic stays in 64 bits; per-row sizes must fit in 32 bits
  if ((int64_t)d.B * (d.gamma + 1) > (int64_t)INT32_MAX) return false;
  return true;
}

WsLayout ws_layout(const dspark_dims& d) {
  WsLayout L;
  const size_t B = (size_t)d.B, G = (size_t)d.gamma, V = (size_t)d.V, r = (size_t)d.r;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t bytes) {
    off = align_up(off, 256);
    const size_t at = off;
    off += bytes;
    return at;
  };
  // regions that depend on (B, gamma) only come first, so that dspark_schedule
  // and dspark_verify find them at the same offsets whatever V, r, H and dtype
  L.sk0 = take(B * G * sizeof(uint32_t));
  L.sk1 = take(B * G * sizeof(uint32_t));
  L.sv0 = take(B * G * sizeof(uint32_t));
  L.sv1 = take(B * G * sizeof(uint32_t));
  L.vrs = take(B * (G + 1) * RS_PARTS * sizeof(float4));
  L.vm = take(B * sizeof(int32_t));
  L.vrowT = take(B * (G + 1) * sizeof(float));
  L.vfmeta = take(B * 4 * sizeof(int32_t));
  L.vfstat = take(B * 4 * sizeof(float));
  L.zh = take(B * G * sizeof(float));
  L.rowstat = take(B * sizeof(float2));
  L.sel = take(B * sizeof(float4));
  // two buffers, positions alternate; fp32-sized so that the RNN head's computed
  // rows fit whatever the dtype
  L.E = take(2 * B * r * sizeof(float));
  L.rnn_s = take(2 * B * r * sizeof(float));  // RNN head state s_{k-1}, s_k
  L.rnn_p = take(B * G * 3 * r * sizeof(float));  // RNN head: W_rnn[:, 2r:] . h_k of every position
  L.rnn_z = take(B * 4 * r * sizeof(uint16_t));     // RNN head, tensor-core recurrent step: z''
  L.rnn_wz = take(3 * r * 4 * r * sizeof(uint16_t));  // its packed weights
  L.rnn_pre = take(B * 3 * r * sizeof(float));      // its products
  const size_t ntiles = (V + kPartialTileMin - 1) / kPartialTileMin;
  // (the fused draft kernel keeps float2 partials of 64-column chunks, rows
  // padded to a multiple of 128)
  const size_t fused_row = ((V + 64 * 128 - 1) / (64 * 128)) * 128 * sizeof(float2);
  L.part = take(B * std::max(ntiles * sizeof(float4), fused_row));
  L.segpart = take(B * kDraftMaxSeg * sizeof(float4));
  // grid-barrier counter, then one tile counter per (sweep, M-tile) (gamma + 1
  // sweeps), then the RNN head's recurrent-unit counters per (position,
  // M-tile); all zeroed by one memset per draft call
  L.gbar = take(16 + (2 * G + 1) * ((B + 127) / 128) * sizeof(uint32_t));
  L.vfin = take(B * 32 * ((((V + 255) / 256) + 31) / 32) * sizeof(float2));
  L.total = align_up(off, 256);
  return L;
}

cudaError_t ensure_smem_limit(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> set_to;  // (device, kernel) -> limit set
  std::lock_guard<std::mutex> lock(mu);
  int& cur = set_to[std::make_pair(dev, func)];
  if (cur >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static dspark_status check_ws(const dspark_dims& d, void* ws, size_t bytes, WsLayout* L) {
  if (!ws || ((uintptr_t)ws & 255u)) return DSPARK_INVALID_ARG;
  *L = ws_layout(d);
  if (bytes < L->total) return DSPARK_INVALID_ARG;
  return DSPARK_OK;
}

// the CUDA error behind the last DSPARK_CUDA_ERROR returned on this thread
static thread_local int t_last_cuda_error = 0;

dspark_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DSPARK_OK;
  t_last_cuda_error = (int)e;
  return DSPARK_CUDA_ERROR;
}

dspark_status check_sched_args(const dspark_sched_args* a, int64_t max_keys) {
  if (!a || a->B < 0 || a->gamma < 1 || a->gamma > DSPARK_MAX_GAMMA) return DSPARK_INVALID_ARG;
  if (a->mode != DSPARK_SCHED_OFF && a->mode != DSPARK_SCHED_GREEDY && a->mode != DSPARK_SCHED_ASYNC_TOPK)
    return DSPARK_INVALID_ARG;
  if ((int64_t)a->B * a->gamma > max_keys) return DSPARK_UNSUPPORTED;
  if (a->B == 0) return DSPARK_OK;
  if (!a->conf_logit || !a->sts_temp || !a->anchor || !a->tokens || !a->ell || !a->offsets || !a->flat_tok ||
      !a->mark_req || !a->mark_pos || !a->n_verify || !a->theta_best)
    return DSPARK_INVALID_ARG;
  if (a->mode != DSPARK_SCHED_OFF && !a->sps) return DSPARK_INVALID_ARG;
  if (a->mode == DSPARK_SCHED_ASYNC_TOPK) {
    if (!a->conf_logit_prev) return DSPARK_INVALID_ARG;
    if (!schedule_async_supported(a->B, a->gamma)) return DSPARK_UNSUPPORTED;
  }
  return DSPARK_OK;
}

}  // namespace dspark

using namespace dspark;

extern "C" {

const char* dspark_status_string(dspark_status s) {
  switch (s) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_INVALID_ARG: return "DSPARK_INVALID_ARG";
    case DSPARK_UNSUPPORTED: return "DSPARK_UNSUPPORTED";
    case DSPARK_CUDA_ERROR: return "DSPARK_CUDA_ERROR";
    case DSPARK_TIMEOUT: return "DSPARK_TIMEOUT";
    case DSPARK_BAD_INPUT: return "DSPARK_BAD_INPUT";
  }
  return "DSPARK_UNKNOWN_STATUS";
}

const char* dspark_version(void) { return "dspark-gb300 0.1 (sm_103a)"; }

uint64_t dspark_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int dspark_last_cuda_error(void) { return t_last_cuda_error; }

dspark_status dspark_workspace_size(const dspark_dims* dims, size_t* bytes) {
  if (!dims || !bytes || !dims_ok(*dims)) return DSPARK_INVALID_ARG;
  *bytes = ws_layout(*dims).total;
  return DSPARK_OK;
}

dspark_status dspark_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < sizeof(WsHeader)) return DSPARK_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), (cudaStream_t)stream));
}

dspark_status dspark_read_error(void* workspace, int32_t* code_host, int32_t* detail_host, void* stream) {
  if (!workspace || !code_host) return DSPARK_INVALID_ARG;
  WsHeader h;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&h, workspace, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return DSPARK_CUDA_ERROR;
  *code_host = h.err_code;
  if (detail_host) *detail_host = h.err_detail;
  e = cudaMemsetAsync(workspace, 0, 2 * sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

// The checks of dspark_draft_sample (B > 0), with the workspace layout.
static dspark_status check_draft_args(const dspark_draft_args* a, void* workspace, size_t workspace_bytes,
                                      WsLayout* L) {
  const dspark_dims& d = a->dims;
  if (!a->U || !a->anchor || !a->temp || !a->req_id || !a->tokens || !a->pd_tok || !a->conf_logit || !a->conf)
    return DSPARK_INVALID_ARG;
  if (!a->pd_rows && (!a->pd_stat || a->head != DSPARK_HEAD_MARKOV)) return DSPARK_INVALID_ARG;
  if (d.r > 0 && (!a->W1 || !a->W2)) return DSPARK_INVALID_ARG;
  if (d.H + d.r > 0 && !a->w) return DSPARK_INVALID_ARG;
  if (d.H > 0 && !a->h) return DSPARK_INVALID_ARG;
  if (a->head != DSPARK_HEAD_MARKOV && a->head != DSPARK_HEAD_RNN) return DSPARK_INVALID_ARG;
  if (a->head == DSPARK_HEAD_RNN && (d.r < 1 || !a->W_rnn)) return DSPARK_INVALID_ARG;
  const void* big[] = {a->U, a->W1, a->W2, a->h, a->w, a->pd_rows, a->head == DSPARK_HEAD_RNN ? a->W_rnn : nullptr};
  for (const void* p : big)
    if (p && !aligned16(p)) return DSPARK_INVALID_ARG;
  return check_ws(d, workspace, workspace_bytes, L);
}

dspark_status dspark_draft_sample(const dspark_draft_args* a, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (!a || !dims_ok(a->dims)) return DSPARK_INVALID_ARG;
  if (a->dims.B == 0) return DSPARK_OK;
  WsLayout L;
  const dspark_status st = check_draft_args(a, workspace, workspace_bytes, &L);
  if (st != DSPARK_OK) return st;
  const cudaError_t e = launch_draft(*a, static_cast<uint8_t*>(workspace), L, (cudaStream_t)stream);
  if (e == cudaErrorNotSupported && !a->pd_rows) return DSPARK_UNSUPPORTED;  // no fused path for the row-free mode
  return cuda_status(e);
}

dspark_status dspark_draft_and_schedule(const dspark_draft_args* da, const dspark_sched_args* sa, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (!da || !dims_ok(da->dims)) return DSPARK_INVALID_ARG;
  const dspark_status chk = check_sched_args(sa, DSPARK_MAX_SCHED_KEYS);
  if (chk != DSPARK_OK) return chk;
  // the schedule reads the draft's confidences and tokens
  if (sa->B != da->dims.B || sa->gamma != da->dims.gamma) return DSPARK_INVALID_ARG;
  if (da->dims.B == 0) return DSPARK_OK;
  if (sa->conf_logit != da->conf_logit || sa->tokens != da->tokens || sa->anchor != da->anchor)
    return DSPARK_INVALID_ARG;
  WsLayout L;
  const dspark_status st = check_draft_args(da, workspace, workspace_bytes, &L);
  if (st != DSPARK_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const cudaStream_t s = (cudaStream_t)stream;
  DraftOverlap ov;
  ov.want = schedule_behind_draft_supported(sa->B, sa->gamma);
  cudaError_t e = launch_draft(*da, ws, L, s, &ov);
  if (e == cudaErrorNotSupported && !da->pd_rows) return DSPARK_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_status(e);
  e = ov.armed ? launch_schedule_behind_draft(*sa, ws, L, ov.sel_done, ov.n_ctas, s) : launch_schedule(*sa, ws, L, s);
  return cuda_status(e);
}

dspark_status dspark_schedule(const dspark_sched_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  const dspark_status chk = check_sched_args(a, DSPARK_MAX_SCHED_KEYS);
  if (chk != DSPARK_OK || a->B == 0) return chk;
  dspark_dims d{a->B, a->gamma, 1, 0, 0, DSPARK_F32};
  WsLayout L;
  const dspark_status st = check_ws(d, workspace, workspace_bytes, &L);
  if (st != DSPARK_OK) return st;
  return cuda_status(launch_schedule(*a, static_cast<uint8_t*>(workspace), L, (cudaStream_t)stream));
}

dspark_status dspark_verify(const dspark_verify_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  if (!a || !dims_ok(a->dims)) return DSPARK_INVALID_ARG;
  const dspark_dims& d = a->dims;
  if (d.B == 0) return DSPARK_OK;
  if (!a->target_logits || !a->offsets || !a->ell || !a->tokens || !a->pd_tok || !a->temp || !a->req_id ||
      !a->n_accept || !a->out_tok || !a->n_out)
    return DSPARK_INVALID_ARG;
  if (a->residual_mode != DSPARK_RESIDUAL_INVERSE_CDF && a->residual_mode != DSPARK_RESIDUAL_REJECTION)
    return DSPARK_INVALID_ARG;
  if (a->residual_mode == DSPARK_RESIDUAL_INVERSE_CDF && !a->pd_rows) return DSPARK_INVALID_ARG;
  if (a->residual_mode == DSPARK_RESIDUAL_REJECTION &&
      (d.r < 1 || !a->U || !a->W1 || !a->W2 || !a->anchor || !a->pd_stat))
    return DSPARK_INVALID_ARG;
  if (!aligned16(a->target_logits) || (a->pd_rows && !aligned16(a->pd_rows))) return DSPARK_INVALID_ARG;
  WsLayout L;
  const dspark_status st = check_ws(d, workspace, workspace_bytes, &L);
  if (st != DSPARK_OK) return st;
  return cuda_status(launch_verify(*a, static_cast<uint8_t*>(workspace), L, (cudaStream_t)stream));
}

dspark_status dspark_pack_rows(const dspark_pack_args* a, void* workspace, void* stream) {
  if (!a || a->V < 1 || a->V > DSPARK_MAX_VOCAB || (a->dtype != DSPARK_BF16 && a->dtype != DSPARK_F32)) return DSPARK_INVALID_ARG;
  if (a->rows_per_request < 1 || a->max_rows < 0 || a->n_src_rows < 0) return DSPARK_INVALID_ARG;
  if (a->max_rows == 0) return DSPARK_OK;
  if (!a->src || !a->mark_req || !a->mark_pos || !a->n_rows || !a->dst) return DSPARK_INVALID_ARG;
  if (workspace && ((uintptr_t)workspace & 255u)) return DSPARK_INVALID_ARG;
  return cuda_status(launch_pack_rows(*a, static_cast<WsHeader*>(workspace), (cudaStream_t)stream));
}

static bool sts_dims_ok(int32_t N, int32_t gamma, int32_t n_grid, int32_t n_bins) {
  if (N < 0 || N > DSPARK_STS_MAX_SAMPLES || gamma < 1 || gamma > DSPARK_MAX_GAMMA) return false;
  if (n_grid < 1 || n_bins < 1) return false;
  return (int64_t)n_bins * std::max<int32_t>(n_grid, 128) <= DSPARK_STS_MAX_TABLE;
}

dspark_status dspark_sts_fit_workspace_size(int32_t N, int32_t gamma, int32_t n_grid, int32_t n_bins,
                                            size_t* bytes) {
  if (!bytes || !sts_dims_ok(N, gamma, n_grid, n_bins)) return DSPARK_INVALID_ARG;
  *bytes = sts_layout(N, gamma, n_grid, n_bins).total;
  return DSPARK_OK;
}

dspark_status dspark_sts_fit(const dspark_sts_fit_args* a, void* workspace, size_t workspace_bytes, void* stream) {
  if (!a || !sts_dims_ok(a->N, a->gamma, a->n_grid, a->n_bins)) return DSPARK_INVALID_ARG;
  if ((a->N > 0 && (!a->conf_logit || !a->accept_len)) || !a->grid || !a->sts_temp || !a->ece)
    return DSPARK_INVALID_ARG;
  if (!workspace || ((uintptr_t)workspace & 255u)) return DSPARK_INVALID_ARG;
  const StsLayout L = sts_layout(a->N, a->gamma, a->n_grid, a->n_bins);
  if (workspace_bytes < L.total) return DSPARK_INVALID_ARG;
  return cuda_status(launch_sts_fit(*a, static_cast<uint8_t*>(workspace), L, (cudaStream_t)stream));
}

}  // extern "C"
