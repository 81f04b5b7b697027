// Packing of the verify batch by the marker tensor.
//
// [DSpark] 补充细节, "高吞吐量与低延迟推理": the kept prefixes of all requests are
// flattened into one buffer with a marker tensor; the SGLang notes on ragged
// verify pack the variable-length requests into a compact buffer before the
// target forward.  Row i of the packed buffer is row (mark_req[i], mark_pos[i])
// of a [R, rows_per_request, V] source, for i < n_rows (a device count, the
// scheduler's n_verify).
//
// One CTA per packed row; the grid covers the largest batch and the CTAs past
// the count return at once, so the launch needs no host round trip.  The
// source may be device memory or pinned host memory the GPU addresses
// directly: then only the kept rows cross the host link.  Rows move in 16-byte
// pieces, four in flight per thread, when the row size and both addresses
// allow it; otherwise element by element.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {

namespace {

constexpr int PK_THREADS = 256;

__global__ void __launch_bounds__(PK_THREADS) k_pack_rows(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                          const int32_t* __restrict__ mark_req,
                                                          const int32_t* __restrict__ mark_pos,
                                                          const int32_t* __restrict__ n_rows, int rows_per_request,
                                                          int64_t n_src_rows, int64_t row_bytes, int esize,
                                                          bool vec16, WsHeader* hdr) {
  const int i = blockIdx.x;
  if (i >= *n_rows) return;
  const int req = mark_req[i], pos = mark_pos[i];
  const int64_t srow = (int64_t)req * rows_per_request + pos;
  if (req < 0 || pos < 0 || pos >= rows_per_request || srow >= n_src_rows) {
    if (threadIdx.x == 0 && hdr) report_error(hdr, DSPARK_BAD_INPUT, i);
    return;
  }
  const uint8_t* s = src + srow * row_bytes;
  uint8_t* d = dst + (int64_t)i * row_bytes;
  if (vec16) {
    const uint4* s4 = reinterpret_cast<const uint4*>(s);
    uint4* d4 = reinterpret_cast<uint4*>(d);
    const int64_t n = row_bytes >> 4;
    int64_t j = threadIdx.x;
    for (; j + 3 * PK_THREADS < n; j += 4 * PK_THREADS) {
      const uint4 a = s4[j], b = s4[j + PK_THREADS], c = s4[j + 2 * PK_THREADS], e = s4[j + 3 * PK_THREADS];
      d4[j] = a;
      d4[j + PK_THREADS] = b;
      d4[j + 2 * PK_THREADS] = c;
      d4[j + 3 * PK_THREADS] = e;
    }
    for (; j < n; j += PK_THREADS) d4[j] = s4[j];
  } else if (esize == 2) {
    const uint16_t* s2 = reinterpret_cast<const uint16_t*>(s);
    uint16_t* d2 = reinterpret_cast<uint16_t*>(d);
    for (int64_t j = threadIdx.x; j < (row_bytes >> 1); j += PK_THREADS) d2[j] = s2[j];
  } else {
    const uint32_t* s1 = reinterpret_cast<const uint32_t*>(s);
    uint32_t* d1 = reinterpret_cast<uint32_t*>(d);
    for (int64_t j = threadIdx.x; j < (row_bytes >> 2); j += PK_THREADS) d1[j] = s1[j];
  }
}

}  // namespace

cudaError_t launch_pack_rows(const dspark_pack_args& a, WsHeader* hdr, cudaStream_t s) {
  const int esize = (int)elem_size(a.dtype);
  const int64_t row_bytes = (int64_t)a.V * esize;
  const bool vec16 = (row_bytes % 16) == 0 && ((uintptr_t)a.src % 16) == 0 && ((uintptr_t)a.dst % 16) == 0;
  k_pack_rows<<<a.max_rows, PK_THREADS, 0, s>>>(static_cast<const uint8_t*>(a.src), static_cast<uint8_t*>(a.dst),
                                                a.mark_req, a.mark_pos, a.n_rows, a.rows_per_request, a.n_src_rows,
                                                row_bytes, esize, vec16, hdr);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dspark
