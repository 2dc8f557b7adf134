// Dispatch of the decode/replay kernels (kda_step.cuh) by state layout and
// projection dtype; each combination is compiled in its own translation unit.
#include "kda_internal.h"
#include "../../include/kda.h"

namespace kda {

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
  if ((int64_t)a.B * a.H * a.layers == 0) return cudaSuccess;
  const bool vk = a.layout == KDA_LAYOUT_VK;
  if (a.dtype == KDA_BF16) return vk ? launch_step_vk_bf16(a, s) : launch_step_kv_bf16(a, s);
  return vk ? launch_step_vk_f32(a, s) : launch_step_kv_f32(a, s);
}

}  // namespace kda
