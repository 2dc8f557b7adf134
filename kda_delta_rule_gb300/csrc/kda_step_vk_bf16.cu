// Decode/replay kernels for bf16 projections and the state stored (dv, dk).
#include "kda_step.cuh"

namespace kda {
cudaError_t launch_step_vk_bf16(const StepArgs& a, cudaStream_t s) { return launch_layout<__nv_bfloat16, true>(a, s); }
}  // namespace kda
