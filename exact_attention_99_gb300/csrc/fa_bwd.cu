// Backward pass of exact attention on sm_103a (placeholder until the
// tcgen05 backward lands).
#include "fa_internal.h"

namespace fa {
cudaError_t launch_bwd(const Problem&, const void*, const float*, const void*, void*, void*, void*, float*, float*,
                       cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace fa
