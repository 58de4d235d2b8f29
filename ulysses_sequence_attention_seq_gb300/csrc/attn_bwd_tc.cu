// attn_bwd_tc.cu -- bf16 attention backward on the tensor cores (in progress).
#include "internal.h"

namespace ulysses {

cudaError_t launch_attn_bwd_tc(const ulysses_problem &, const TmaEncoder &, const void *,
                               const void *, const void *, const void *, const float *,
                               const float *, const void *, void *, void *, void *, uint32_t *,
                               cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ulysses
