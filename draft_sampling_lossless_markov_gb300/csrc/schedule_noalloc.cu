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

#include "common.cuh"
#include "dspark.h"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kNoallocKeys = DSPARK_MAX_SCHED_KEYS;  // candidates (B * gamma) per call, at most

// 4 x 65536 x 4 bytes = 1 MiB, present in every GPU context that loads the
// library until the process exits.  Layout: keys copy 0, keys copy 1, values
// copy 0, values copy 1.  Host code must not use this name as a device
// address: it refers to a host-side stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint32_t g_sched_scratch[4 * kNoallocKeys];

// Device address of g_sched_scratch in the current device's context.  The
// lookup allocates nothing and runs on every call, so the address always
// belongs to the context that is current now: a process that resets the
// device (which reloads the library's module and may move the array), or a
// caller that makes its own driver-API context current on the GPU, gets that
// context's copy rather than a stale one.  The first lookup in a context can
// load the library's device code there, which is why the first call on a
// device should come before any stream capture.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_sched_scratch);
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" dspark_status dspark_schedule_noalloc(const dspark_sched_args* a, void* stream) {
  // the checks of dspark_schedule, with the static array's capacity as the limit
  const dspark_status chk = check_sched_args(a, kNoallocKeys);
  if (chk != DSPARK_OK || a->B == 0) return chk;

  void* scratch = nullptr;
  const dspark_status st = cuda_status(scratch_address(&scratch));
  if (st != DSPARK_OK) return st;
  // The kernel writes every key and value it later reads (all B * gamma of
  // them, in every sort pass), so nothing left from an earlier call needs
  // clearing.
  WsLayout L;
  L.sk0 = 0;
  L.sk1 = (size_t)kNoallocKeys * sizeof(uint32_t);
  L.sv0 = 2 * (size_t)kNoallocKeys * sizeof(uint32_t);
  L.sv1 = 3 * (size_t)kNoallocKeys * sizeof(uint32_t);
  L.total = 4 * (size_t)kNoallocKeys * sizeof(uint32_t);
  return cuda_status(launch_schedule(*a, static_cast<uint8_t*>(scratch), L, (cudaStream_t)stream));
}
