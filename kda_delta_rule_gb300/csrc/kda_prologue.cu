// Dispatch of the input-prologue kernels (kda_prologue.cuh) by dtype; each dtype is
// compiled in its own translation unit.
#include "kda_internal.h"
#include "../../include/kda.h"

namespace kda {

cudaError_t launch_prologue(const ProArgs& a, const ProSched& sched, cudaStream_t s) {
  if (a.w < 2 || a.w > 8) return cudaErrorInvalidValue;
  return a.dtype == KDA_BF16 ? launch_prologue_bf16(a, sched, s) : launch_prologue_f32(a, sched, s);
}

int read_and_clear_prologue_errors(int* flags) {
  const int e = read_and_clear_prologue_errors_f32(flags);
  return e != 0 ? e : read_and_clear_prologue_errors_bf16(flags);
}

}  // namespace kda
