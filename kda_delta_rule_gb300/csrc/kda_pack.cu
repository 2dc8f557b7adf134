// pack_heads / unpack_heads (KIMI K3 Serve demo page, §1.5 unified page pool
// and Tab 7 store_kda / load_kda): (B,H,dk,dv) fp32 states <-> one flat,
// head-contiguous buffer, zero-padded past the state.  Bit-exact 128-bit
// copies; the (b,h) blocks of the source may be strided (e.g. one slot of a
// batched decode state buffer).
#include "kda_internal.h"

namespace kda {
namespace {

__global__ void pack_kernel(const float* __restrict__ S, int64_t stride_b, int64_t stride_h,
                            float* __restrict__ flat, int64_t flat_elems, int H,
                            int64_t head_elems, int64_t n_heads) {
  const int64_t n4 = n_heads * head_elems / 4;
  const int64_t h4 = head_elems / 4;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n4; t += step) {
    const int64_t head = t / h4, e = (t - head * h4) * 4;
    const int64_t b = head / H, h = head - b * H;
    float4 x = *reinterpret_cast<const float4*>(S + b * stride_b + h * stride_h + e);
    *reinterpret_cast<float4*>(flat + t * 4) = x;
  }
  // zero tail of the page
  for (int64_t t = n_heads * head_elems + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
       t < flat_elems; t += step)
    flat[t] = 0.f;
}

__global__ void unpack_kernel(const float* __restrict__ flat, float* __restrict__ S,
                              int64_t stride_b, int64_t stride_h, int H, int64_t head_elems,
                              int64_t n_heads) {
  const int64_t n4 = n_heads * head_elems / 4;
  const int64_t h4 = head_elems / 4;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n4; t += step) {
    const int64_t head = t / h4, e = (t - head * h4) * 4;
    const int64_t b = head / H, h = head - b * H;
    float4 x = *reinterpret_cast<const float4*>(flat + t * 4);
    *reinterpret_cast<float4*>(S + b * stride_b + h * stride_h + e) = x;
  }
}

unsigned grid_for(int64_t n4) {
  int64_t g = (n4 + 255) / 256;
  const int64_t cap = 152 * 16;   // enough resident CTAs to saturate HBM
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (unsigned)g;
}

}  // namespace

cudaError_t launch_pack(const float* S, int64_t stride_b, int64_t stride_h, float* flat,
                        int64_t flat_elems, int B, int H, int dk, int dv, cudaStream_t s) {
  const int64_t head_elems = (int64_t)dk * dv, n_heads = (int64_t)B * H;
  if (flat_elems == 0) return cudaSuccess;
  int64_t work = n_heads * head_elems / 4;
  int64_t tail = flat_elems - n_heads * head_elems;
  if (tail > work) work = tail;
  pack_kernel<<<grid_for(work), 256, 0, s>>>(S, stride_b, stride_h, flat, flat_elems, H,
                                              head_elems, n_heads);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const float* flat, float* S, int64_t stride_b, int64_t stride_h,
                          int B, int H, int dk, int dv, cudaStream_t s) {
  const int64_t head_elems = (int64_t)dk * dv, n_heads = (int64_t)B * H;
  if (n_heads == 0) return cudaSuccess;
  unpack_kernel<<<grid_for(n_heads * head_elems / 4), 256, 0, s>>>(flat, S, stride_b, stride_h,
                                                                   H, head_elems, n_heads);
  return cudaGetLastError();
}

}  // namespace kda
