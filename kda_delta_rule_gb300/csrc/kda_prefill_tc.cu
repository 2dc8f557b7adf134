// Tensor-core (tcgen05) chunked prefill: not built yet; every call falls
// through to the fp32 CUDA-core kernel.
#include "kda_internal.h"

namespace kda {
cudaError_t launch_prefill_tc(const PrefillArgs&, const PrefillSched&, cudaStream_t, bool* handled) {
  *handled = false;
  return cudaSuccess;
}
}  // namespace kda
