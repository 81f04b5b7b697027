// Tensor-core (tcgen05) logits passes of the draft sampler.
#include "common.cuh"
#include "internal.h"

namespace dspark {

bool draft_tc_supported(const dspark_dims&) { return false; }

cudaError_t launch_draft_tc_pass(const dspark_draft_args&, uint8_t*, const WsLayout&, int, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace dspark
