// dspark_schedule_noalloc: the prefix scheduler with its scratch memory in a
// fixed array compiled into the library, for callers that cannot allocate
// device memory (see the declaration in dspark.h for who they are).
//
// The scheduler kernel sorts up to DSPARK_MAX_SCHED_KEYS candidates through
// two key buffers and two value buffers.  Here those four buffers live in one
// file-scope device array instead of the caller's workspace.  The kernel and
// its launcher are the ones dspark_schedule uses; only the scratch address
// differs.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "dspark.h"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kNoallocKeys = DSPARK_MAX_SCHED_KEYS;  // candidates (B * gamma) per call, at most
constexpr int kMaxDevices = 64;

// 4 x 65536 x 4 bytes = 1 MiB, present in every GPU context that loads the
// library until the process exits.  Layout: keys copy 0, keys copy 1, values
// copy 0, values copy 1.  Host code must not use this name as a device
// address: it refers to a host-side stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint32_t g_sched_scratch[4 * kNoallocKeys];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of g_sched_scratch on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sched_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" dspark_status dspark_schedule_noalloc(const dspark_sched_args* a, void* stream) {
  // the same argument checks as dspark_schedule
  if (!a || a->B < 0 || a->gamma < 1 || a->gamma > DSPARK_MAX_GAMMA) return DSPARK_INVALID_ARG;
  if (a->mode != DSPARK_SCHED_OFF && a->mode != DSPARK_SCHED_GREEDY && a->mode != DSPARK_SCHED_ASYNC_TOPK)
    return DSPARK_INVALID_ARG;
  if ((int64_t)a->B * a->gamma > kNoallocKeys) return DSPARK_UNSUPPORTED;  // beyond the static array
  if (a->B == 0) return DSPARK_OK;
  if (!a->conf_logit || !a->sts_temp || !a->anchor || !a->tokens || !a->ell || !a->offsets || !a->flat_tok ||
      !a->mark_req || !a->mark_pos || !a->n_verify || !a->theta_best)
    return DSPARK_INVALID_ARG;
  if (a->mode != DSPARK_SCHED_OFF && !a->sps) return DSPARK_INVALID_ARG;
  if (a->mode == DSPARK_SCHED_ASYNC_TOPK) {
    if (!a->conf_logit_prev) return DSPARK_INVALID_ARG;
    if (!schedule_async_supported(a->B, a->gamma)) return DSPARK_UNSUPPORTED;
  }

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return DSPARK_CUDA_ERROR;
  // The kernel writes every key and value it later reads (all B * gamma of
  // them, in every sort pass), so nothing left from an earlier call needs
  // clearing.
  WsLayout L;
  L.sk0 = 0;
  L.sk1 = (size_t)kNoallocKeys * sizeof(uint32_t);
  L.sv0 = 2 * (size_t)kNoallocKeys * sizeof(uint32_t);
  L.sv1 = 3 * (size_t)kNoallocKeys * sizeof(uint32_t);
  L.total = 4 * (size_t)kNoallocKeys * sizeof(uint32_t);
  const cudaError_t e = launch_schedule(*a, static_cast<uint8_t*>(scratch), L, (cudaStream_t)stream);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_CUDA_ERROR;
}
