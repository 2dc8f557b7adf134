// Raw-input ring: the streaming window of raw draft projections that a commit
// replays (fold-every-commit), kept in device memory the caller provides.
//
// The stored steps are laid out exactly as the draft-projection cache the
// replay kernel reads, [capacity][B][H][D] per tensor, so a commit replays
// straight from the ring: step s of the window is stored step
// (oldest + s) mod capacity, an offset the replay kernel applies while it
// stages the projections.  Pushing one step is five device-to-device copies.
#include <cuda_runtime.h>

#include <cstdio>

#include "../../include/kda.h"
#include "kda_internal.h"

struct kda_raw_ring {
  char* base;
  int capacity, B, H, dk, dv, dtype;
  int64_t off_q, off_k, off_g, off_v, off_beta;   // byte offsets of the five arrays
  int64_t pushed;                                 // pushes since the last reset
};

namespace {

int64_t up256(int64_t x) { return (x + 255) / 256 * 256; }

int64_t step_elems_k(const kda_raw_ring* r) { return (int64_t)r->B * r->H * r->dk; }
int64_t step_elems_v(const kda_raw_ring* r) { return (int64_t)r->B * r->H * r->dv; }
int64_t step_elems_b(const kda_raw_ring* r) { return (int64_t)r->B * r->H; }
int64_t es_of(int dtype) { return dtype == KDA_BF16 ? 2 : 4; }

int ring_len(const kda_raw_ring* r) { return (int)(r->pushed < r->capacity ? r->pushed : r->capacity); }
int ring_oldest(const kda_raw_ring* r) { return r->pushed <= r->capacity ? 0 : (int)(r->pushed % r->capacity); }

int cuda_fail(cudaError_t e, const char* what) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  return kda::set_error(KDA_ERR_CUDA, msg);
}

bool bad_dims(int capacity, int B, int H, int dk, int dv, int dtype) {
  return capacity < 1 || capacity > KDA_MAX_DRAFT || B < 1 || H < 1 || !(dk == 32 || dk == 64 || dk == 128) ||
         !(dv == 32 || dv == 64 || dv == 128) || (dtype != KDA_F32 && dtype != KDA_BF16);
}

}  // namespace

extern "C" int64_t kda_ring_bytes(int capacity, int B, int H, int dk, int dv, int dtype) {
  if (bad_dims(capacity, B, H, dk, dv, dtype))
    return kda::set_error(KDA_ERR_SHAPE, "kda_ring_bytes: capacity in [1, KDA_MAX_DRAFT], B, H >= 1, "
                                         "dk, dv in {32, 64, 128}, dtype f32 or bf16");
  const int64_t es = es_of(dtype), n = (int64_t)capacity * B * H;
  return 3 * up256(n * dk * es) + up256(n * dv * es) + up256(n * es);
}

extern "C" int kda_ring_create(void* device_base, int capacity, int B, int H, int dk, int dv, int dtype,
                               kda_raw_ring** ring_out) {
  if (!ring_out) return kda::set_error(KDA_ERR_ARG, "kda_ring_create: ring_out is NULL");
  *ring_out = nullptr;
  const int64_t bytes = kda_ring_bytes(capacity, B, H, dk, dv, dtype);
  if (bytes < 0) return (int)bytes;
  if (!device_base) return kda::set_error(KDA_ERR_ARG, "kda_ring_create: device_base is NULL");
  if (((uintptr_t)device_base & 255) != 0) return kda::set_error(KDA_ERR_ALIGN, "device_base must be 256-byte aligned");
  kda_raw_ring* r = new kda_raw_ring;
  r->base = static_cast<char*>(device_base);
  r->capacity = capacity; r->B = B; r->H = H; r->dk = dk; r->dv = dv; r->dtype = dtype;
  const int64_t es = es_of(dtype), n = (int64_t)capacity * B * H;
  r->off_q = 0;
  r->off_k = r->off_q + up256(n * dk * es);
  r->off_g = r->off_k + up256(n * dk * es);
  r->off_v = r->off_g + up256(n * dk * es);
  r->off_beta = r->off_v + up256(n * dv * es);
  r->pushed = 0;
  *ring_out = r;
  return kda::set_error(KDA_OK, "");
}

extern "C" int kda_ring_destroy(kda_raw_ring* ring) {
  delete ring;
  return KDA_OK;
}

extern "C" int kda_ring_reset(kda_raw_ring* ring) {
  if (!ring) return kda::set_error(KDA_ERR_ARG, "kda_ring_reset: ring is NULL");
  ring->pushed = 0;
  return KDA_OK;
}

extern "C" int kda_ring_len(const kda_raw_ring* ring) {
  if (!ring) return kda::set_error(KDA_ERR_ARG, "kda_ring_len: ring is NULL");
  return ring_len(ring);
}

extern "C" int kda_ring_push(kda_raw_ring* ring, const void* q, const void* k, const void* v, const void* g,
                             const void* beta, kda_stream_t stream) {
  if (!ring) return kda::set_error(KDA_ERR_ARG, "kda_ring_push: ring is NULL");
  if (!q || !k || !v || !g || !beta) return kda::set_error(KDA_ERR_ARG, "kda_ring_push: null projection pointer");
  const int slot = (int)(ring->pushed % ring->capacity);   // the oldest step once the ring is full
  const int64_t es = es_of(ring->dtype);
  const int64_t nk = step_elems_k(ring) * es, nv = step_elems_v(ring) * es, nb = step_elems_b(ring) * es;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(ring->base + ring->off_q + slot * nk, q, nk, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ring->base + ring->off_k + slot * nk, k, nk, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ring->base + ring->off_g + slot * nk, g, nk, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ring->base + ring->off_v + slot * nv, v, nv, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ring->base + ring->off_beta + slot * nb, beta, nb, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "kda_ring_push");
  ++ring->pushed;
  return kda::set_error(KDA_OK, "");
}

extern "C" int kda_ring_window(const kda_raw_ring* ring, void* q, void* k, void* v, void* g, void* beta,
                               kda_stream_t stream) {
  if (!ring) return kda::set_error(KDA_ERR_ARG, "kda_ring_window: ring is NULL");
  const int len = ring_len(ring);
  if (len == 0) return KDA_OK;
  if (!q || !k || !v || !g || !beta) return kda::set_error(KDA_ERR_ARG, "kda_ring_window: null output pointer");
  const int old = ring_oldest(ring), first = ring->capacity - old < len ? ring->capacity - old : len;
  const int64_t es = es_of(ring->dtype);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  auto two_runs = [&](void* dst, int64_t off, int64_t step_bytes) {
    char* d = static_cast<char*>(dst);
    const char* src = ring->base + off;
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(d, src + old * step_bytes, first * step_bytes, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && len > first)
      e = cudaMemcpyAsync(d + first * step_bytes, src, (len - first) * step_bytes, cudaMemcpyDeviceToDevice, s);
  };
  two_runs(q, ring->off_q, step_elems_k(ring) * es);
  two_runs(k, ring->off_k, step_elems_k(ring) * es);
  two_runs(g, ring->off_g, step_elems_k(ring) * es);
  two_runs(v, ring->off_v, step_elems_v(ring) * es);
  two_runs(beta, ring->off_beta, step_elems_b(ring) * es);
  if (e != cudaSuccess) return cuda_fail(e, "kda_ring_window");
  return kda::set_error(KDA_OK, "");
}

extern "C" int kda_verify_replay_ring(const kda_raw_ring* ring, const float* S_committed,
                                      const int32_t* n_accepted, float* S_new, void* out, int mode,
                                      kda_stream_t stream) {
  if (!ring) return kda::set_error(KDA_ERR_ARG, "kda_verify_replay_ring: ring is NULL");
  if (mode != KDA_MODE_DECAY_FIRST && mode != KDA_MODE_UNDECAYED_DELTA)
    return kda::set_error(KDA_ERR_ARG, "kda_verify_replay_ring: bad mode");
  const int len = ring_len(ring);
  if (len == 0) return kda::set_error(KDA_ERR_SHAPE, "kda_verify_replay_ring: the window is empty");
  if (!S_committed || !n_accepted || !S_new || !out)
    return kda::set_error(KDA_ERR_ARG, "kda_verify_replay_ring: null pointer argument");
  if (((uintptr_t)S_committed & 15) || ((uintptr_t)S_new & 15) || ((uintptr_t)out & 15))
    return kda::set_error(KDA_ERR_ALIGN, "state and output pointers must be 16-byte aligned");
  const int64_t heads = (int64_t)ring->B * ring->H, sbytes = heads * ring->dk * ring->dv * 4;
  const char* a0 = reinterpret_cast<const char*>(S_committed);
  const char* a1 = reinterpret_cast<const char*>(S_new);
  if (a0 < a1 + sbytes && a1 < a0 + sbytes)
    return kda::set_error(KDA_ERR_ALIAS, "S_new overlaps S_committed: the committed state must not be written");
  kda::StepArgs a{};
  a.S_in = S_committed; a.S_out = S_new;
  a.q = ring->base + ring->off_q; a.k = ring->base + ring->off_k; a.v = ring->base + ring->off_v;
  a.g = ring->base + ring->off_g; a.beta = ring->base + ring->off_beta;
  a.out = out;
  a.n_accepted = n_accepted;
  a.B = ring->B; a.H = ring->H; a.dk = ring->dk; a.dv = ring->dv; a.steps = len;
  a.dtype = ring->dtype; a.mode = mode;
  a.layers = 1; a.proj_steps = ring->capacity; a.ring_start = ring_oldest(ring);
  a.out_head_stride = (int64_t)len * ring->dv; a.out_step_stride = ring->dv;
  cudaError_t e = kda::launch_step(a, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kda_verify_replay_ring launch");
  return kda::set_error(KDA_OK, "");
}
