// Decode/replay kernels for f32 projections and the state stored (dv, dk).
#include "kda_step.cuh"

namespace kda {
cudaError_t launch_step_vk_f32(const StepArgs& a, cudaStream_t s) { return launch_layout<float, true>(a, s); }
}  // namespace kda
