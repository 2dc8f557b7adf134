// Decode/replay kernels for bf16 projections and the state stored (dk, dv).
#include "kda_step.cuh"

namespace kda {
cudaError_t launch_step_kv_bf16(const StepArgs& a, cudaStream_t s) { return launch_layout<__nv_bfloat16, false>(a, s); }
}  // namespace kda
