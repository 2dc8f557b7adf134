// Decode/replay kernels for f32 projections and the state stored (dk, dv).
#include "kda_step.cuh"

namespace kda {
cudaError_t launch_step_kv_f32(const StepArgs& a, cudaStream_t s) { return launch_layout<float, false>(a, s); }
}  // namespace kda
