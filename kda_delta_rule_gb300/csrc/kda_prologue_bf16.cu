// Input prologue kernels for bf16 inputs and outputs.
#include "kda_prologue.cuh"

namespace kda {
cudaError_t launch_prologue_bf16(const ProArgs& a, const ProSched& sched, cudaStream_t s) {
  return launch_t<__nv_bfloat16>(a, sched, s);
}

int read_and_clear_prologue_errors_bf16(int* flags) {
  int word = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&word, tc::g_kda_device_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(tc::g_kda_device_error, &zero, sizeof(int));
  *flags |= word;
  return (int)e;
}
}  // namespace kda
