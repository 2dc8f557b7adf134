// C ABI of the KDA library: host-side validation, scheduling and dispatch,
// plus the unified page pool.  Every check runs before any launch, so a call
// that returns an error has launched nothing and written nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <numeric>
#include <set>
#include <string>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace kda {
cudaError_t launch_prefill_simt(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s);
cudaError_t launch_prefill_tc(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s,
                              bool* handled);
}  // namespace kda

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int ok() {
  g_last_error.clear();
  return KDA_OK;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool head_dim_ok(int d) { return d == 32 || d == 64 || d == 128; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t elem_size(int dtype) { return dtype == KDA_BF16 ? 2 : 4; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  auto pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

int check_common(int dk, int dv, int dtype, int mode) {
  if (dtype != KDA_F32 && dtype != KDA_BF16) return fail(KDA_ERR_DTYPE, "dtype %d is not KDA_F32 or KDA_BF16", dtype);
  if (mode != KDA_MODE_DECAY_FIRST && mode != KDA_MODE_UNDECAYED_DELTA)
    return fail(KDA_ERR_ARG, "mode %d is not a KDA_MODE_*", mode);
  if (!head_dim_ok(dk) || !head_dim_ok(dv))
    return fail(KDA_ERR_SHAPE, "head sizes dk=%d dv=%d: each must be 32, 64 or 128", dk, dv);
  return KDA_OK;
}

}  // namespace

namespace kda {
namespace {
std::atomic<int> g_chain_columns{0};
}  // namespace
int prefill_chain_columns() { return g_chain_columns.load(std::memory_order_relaxed); }
}  // namespace kda

extern "C" {

int kda_version(void) { return 1; }

const char* kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_ARG: return "KDA_ERR_ARG";
    case KDA_ERR_SHAPE: return "KDA_ERR_SHAPE";
    case KDA_ERR_DTYPE: return "KDA_ERR_DTYPE";
    case KDA_ERR_ALIGN: return "KDA_ERR_ALIGN";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_NOMEM: return "KDA_ERR_NOMEM";
    case KDA_ERR_ALIAS: return "KDA_ERR_ALIAS";
  }
  return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error(void) { return g_last_error.c_str(); }

// ---------------------------------------------------------------------------
int kda_decode_step(float* S, const void* q, const void* k, const void* v, const void* g,
                    const void* beta, void* o, int B, int H, int dk, int dv, int dtype, int mode,
                    kda_stream_t stream) {
  if (int st = check_common(dk, dv, dtype, mode)) return st;
  if (B < 0 || H < 0) return fail(KDA_ERR_SHAPE, "negative B=%d or H=%d", B, H);
  const int64_t heads = (int64_t)B * H;
  if (heads == 0) return ok();
  if (heads > 0x7fffffffLL) return fail(KDA_ERR_SHAPE, "B*H too large");
  if (!S || !q || !k || !v || !g || !beta || !o) return fail(KDA_ERR_ARG, "null pointer argument");
  if (!aligned16(S) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(o))
    return fail(KDA_ERR_ALIGN, "state, projection and output pointers must be 16-byte aligned");
  const size_t es = elem_size(dtype);
  if (overlap(o, heads * dv * es, S, heads * dk * dv * 4))
    return fail(KDA_ERR_ALIAS, "o overlaps the state");
  kda::StepArgs a{};
  a.S_in = S; a.S_out = S;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = o;
  a.n_accepted = nullptr;
  a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.steps = 1; a.dtype = dtype; a.mode = mode;
  a.layers = 1; a.proj_steps = 1; a.ring_start = 0;
  a.out_head_stride = dv; a.out_step_stride = 0;
  return cuda_status(kda::launch_step(a, reinterpret_cast<cudaStream_t>(stream)), "kda_decode_step launch");
}

// ---------------------------------------------------------------------------
int kda_verify_replay_layers(int layers, const float* S_committed, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, const int32_t* n_accepted, float* S_new,
                             void* out, int draft, int B, int H, int dk, int dv, int dtype, int mode,
                             kda_stream_t stream) {
  if (int st = check_common(dk, dv, dtype, mode)) return st;
  if (layers < 0 || B < 0 || H < 0) return fail(KDA_ERR_SHAPE, "negative layers=%d, B=%d or H=%d", layers, B, H);
  if (draft < 1 || draft > KDA_MAX_DRAFT)
    return fail(KDA_ERR_SHAPE, "draft=%d outside [1, %d]", draft, KDA_MAX_DRAFT);
  const int64_t heads = (int64_t)layers * B * H;
  if (heads == 0) return ok();
  if (heads > 0x7fffffffLL) return fail(KDA_ERR_SHAPE, "layers*B*H too large");
  if (!S_committed || !q || !k || !v || !g || !beta || !n_accepted || !S_new || !out)
    return fail(KDA_ERR_ARG, "null pointer argument");
  if (!aligned16(S_committed) || !aligned16(S_new) || !aligned16(q) || !aligned16(k) ||
      !aligned16(v) || !aligned16(g) || !aligned16(out))
    return fail(KDA_ERR_ALIGN, "state, projection and output pointers must be 16-byte aligned");
  const size_t sbytes = heads * dk * dv * 4;
  const size_t es = elem_size(dtype);
  if (overlap(S_new, sbytes, S_committed, sbytes))
    return fail(KDA_ERR_ALIAS, "S_new overlaps S_committed: the committed state must not be written");
  if (overlap(out, heads * draft * dv * es, S_committed, sbytes) ||
      overlap(out, heads * draft * dv * es, S_new, sbytes))
    return fail(KDA_ERR_ALIAS, "out overlaps a state buffer");
  kda::StepArgs a{};
  a.S_in = S_committed; a.S_out = S_new;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out;
  a.n_accepted = n_accepted;
  a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.steps = draft; a.dtype = dtype; a.mode = mode;
  a.layers = layers; a.proj_steps = draft; a.ring_start = 0;
  a.out_head_stride = (int64_t)draft * dv; a.out_step_stride = dv;
  return cuda_status(kda::launch_step(a, reinterpret_cast<cudaStream_t>(stream)), "kda_verify_replay launch");
}

int kda_verify_replay(const float* S_committed, const void* q, const void* k, const void* v,
                      const void* g, const void* beta, const int32_t* n_accepted, float* S_new,
                      void* out, int draft, int B, int H, int dk, int dv, int dtype, int mode,
                      kda_stream_t stream) {
  return kda_verify_replay_layers(1, S_committed, q, k, v, g, beta, n_accepted, S_new, out, draft, B, H, dk, dv,
                                  dtype, mode, stream);
}

// ---------------------------------------------------------------------------
static int check_slots(int64_t n_slots, int layout, const int32_t* slot_ids) {
  if (layout != KDA_LAYOUT_KV && layout != KDA_LAYOUT_VK) return fail(KDA_ERR_ARG, "layout=%d is not a KDA_LAYOUT_*", layout);
  if (n_slots < 1) return fail(KDA_ERR_SHAPE, "n_slots=%lld, must be >= 1", (long long)n_slots);
  if (!slot_ids) return fail(KDA_ERR_ARG, "slot ids are NULL");
  return KDA_OK;
}

int kda_decode_step_slots(float* S_pool, int64_t n_slots, const int32_t* slot_ids, int layout, const void* q,
                          const void* k, const void* v, const void* g, const void* beta, void* o, int B, int H,
                          int dk, int dv, int dtype, int mode, kda_stream_t stream) {
  if (int st = check_common(dk, dv, dtype, mode)) return st;
  if (B < 0 || H < 0) return fail(KDA_ERR_SHAPE, "negative B=%d or H=%d", B, H);
  const int64_t heads = (int64_t)B * H;
  if (heads == 0) return ok();
  if (heads > 0x7fffffffLL) return fail(KDA_ERR_SHAPE, "B*H too large");
  if (int st = check_slots(n_slots, layout, slot_ids)) return st;
  if (n_slots > (int64_t)1 << 40) return fail(KDA_ERR_SHAPE, "n_slots too large");
  if (!S_pool || !q || !k || !v || !g || !beta || !o) return fail(KDA_ERR_ARG, "null pointer argument");
  if (!aligned16(S_pool) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(o))
    return fail(KDA_ERR_ALIGN, "state, projection and output pointers must be 16-byte aligned");
  const size_t es = elem_size(dtype);
  if (overlap(o, heads * dv * es, S_pool, (size_t)n_slots * H * dk * dv * 4))
    return fail(KDA_ERR_ALIAS, "o overlaps the state pool");
  kda::StepArgs a{};
  a.S_in = S_pool; a.S_out = S_pool;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = o;
  a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.steps = 1; a.dtype = dtype; a.mode = mode;
  a.layers = 1; a.proj_steps = 1; a.ring_start = 0;
  a.out_head_stride = dv; a.out_step_stride = 0;
  a.slot_in = slot_ids; a.slot_out = slot_ids; a.n_slots = n_slots; a.layout = layout;
  return cuda_status(kda::launch_step(a, reinterpret_cast<cudaStream_t>(stream)), "kda_decode_step_slots launch");
}

int kda_decode_step_fused(float* S, int64_t n_slots, const int32_t* slot_ids, int layout, void* conv_state,
                          const void* mixed_qkv, const void* conv_weight, int w, const void* g_logits,
                          const void* beta_logits, float g_min, int act, void* o, void* q_out, void* k_out,
                          void* v_out, void* g_out, void* beta_out, int B, int H, int dk, int dv, int dtype,
                          int mode, kda_stream_t stream) {
  if (int st = check_common(dk, dv, dtype, mode)) return st;
  if (B < 0 || H < 0) return fail(KDA_ERR_SHAPE, "negative B=%d or H=%d", B, H);
  const int64_t heads = (int64_t)B * H;
  if (heads == 0) return ok();
  if (heads > 0x7fffffffLL) return fail(KDA_ERR_SHAPE, "B*H too large");
  if (layout != KDA_LAYOUT_KV && layout != KDA_LAYOUT_VK) return fail(KDA_ERR_ARG, "layout=%d is not a KDA_LAYOUT_*", layout);
  if (slot_ids && (n_slots < 1 || n_slots > ((int64_t)1 << 40)))
    return fail(KDA_ERR_SHAPE, "n_slots=%lld outside [1, 2^40]", (long long)n_slots);
  if (w < 2 || w > 4) return fail(KDA_ERR_SHAPE, "conv kernel size w=%d outside [2, 4] (fused decode)", w);
  if (act != KDA_ACT_NONE && act != KDA_ACT_SILU) return fail(KDA_ERR_ARG, "act=%d is not a KDA_ACT_*", act);
  if (!(g_min < 0.f)) return fail(KDA_ERR_ARG, "g_min=%g must be negative", (double)g_min);
  if (!S || !conv_state || !mixed_qkv || !conv_weight || !g_logits || !beta_logits || !o)
    return fail(KDA_ERR_ARG, "null pointer argument");
  const int n_keep = (q_out != nullptr) + (k_out != nullptr) + (v_out != nullptr) + (g_out != nullptr) +
                     (beta_out != nullptr);
  if (n_keep != 0 && n_keep != 5) return fail(KDA_ERR_ARG, "q_out, k_out, v_out, g_out, beta_out: give all or none");
  const void* al[] = {S, conv_state, mixed_qkv, conv_weight, g_logits, beta_logits, o, q_out, k_out, v_out, g_out, beta_out};
  for (const void* ptr : al)
    if (ptr && !aligned16(ptr)) return fail(KDA_ERR_ALIGN, "pointers must be 16-byte aligned");
  const size_t es = elem_size(dtype), C = (size_t)H * (2 * dk + dv);
  const size_t rows = slot_ids ? (size_t)n_slots : (size_t)B;
  const void* bufs[] = {S, conv_state, mixed_qkv, conv_weight, g_logits, beta_logits, o, q_out, k_out, v_out, g_out, beta_out};
  const size_t bytes[] = {rows * H * dk * dv * 4, rows * (w - 1) * C * es, (size_t)B * C * es, C * w * es,
                          (size_t)heads * dk * es, (size_t)heads * es, (size_t)heads * dv * es, (size_t)heads * dk * es,
                          (size_t)heads * dk * es, (size_t)heads * dv * es, (size_t)heads * dk * es, (size_t)heads * es};
  for (int i = 0; i < 12; ++i)
    for (int j = 0; j < i; ++j)
      if (overlap(bufs[i], bytes[i], bufs[j], bytes[j])) return fail(KDA_ERR_ALIAS, "two arguments overlap");
  kda::StepArgs a{};
  a.S_in = S; a.S_out = S;
  a.out = o;
  a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.steps = 1; a.dtype = dtype; a.mode = mode;
  a.layers = 1; a.proj_steps = 1; a.ring_start = 0;
  a.out_head_stride = dv; a.out_step_stride = 0;
  a.slot_in = slot_ids; a.slot_out = slot_ids; a.n_slots = n_slots; a.layout = layout;
  a.mixed = mixed_qkv; a.conv_state = conv_state; a.conv_w = conv_weight;
  a.g_logits = g_logits; a.beta_logits = beta_logits;
  a.q_out = q_out; a.k_out = k_out; a.v_out = v_out; a.g_out = g_out; a.beta_out = beta_out;
  a.conv_size = w; a.act = act; a.g_min = g_min; a.eps = 1e-6f;
  return cuda_status(kda::launch_step(a, reinterpret_cast<cudaStream_t>(stream)), "kda_decode_step_fused launch");
}

int kda_verify_replay_slots(int layers, const float* S_pool, float* S_pool_new, int64_t n_slots,
                            const int32_t* slot_in, const int32_t* slot_out, int layout, const void* q,
                            const void* k, const void* v, const void* g, const void* beta,
                            const int32_t* n_accepted, void* out, int draft, int B, int H, int dk, int dv,
                            int dtype, int mode, kda_stream_t stream) {
  if (int st = check_common(dk, dv, dtype, mode)) return st;
  if (layers < 0 || B < 0 || H < 0) return fail(KDA_ERR_SHAPE, "negative layers=%d, B=%d or H=%d", layers, B, H);
  if (draft < 1 || draft > KDA_MAX_DRAFT)
    return fail(KDA_ERR_SHAPE, "draft=%d outside [1, %d]", draft, KDA_MAX_DRAFT);
  const int64_t heads = (int64_t)layers * B * H;
  if (heads == 0) return ok();
  if (heads > 0x7fffffffLL) return fail(KDA_ERR_SHAPE, "layers*B*H too large");
  if (int st = check_slots(n_slots, layout, slot_in)) return st;
  if (n_slots > (int64_t)1 << 40) return fail(KDA_ERR_SHAPE, "n_slots too large");
  if (!S_pool || !S_pool_new || !q || !k || !v || !g || !beta || !n_accepted || !out)
    return fail(KDA_ERR_ARG, "null pointer argument");
  if (!aligned16(S_pool) || !aligned16(S_pool_new) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(g) || !aligned16(out))
    return fail(KDA_ERR_ALIGN, "state, projection and output pointers must be 16-byte aligned");
  const size_t pbytes = (size_t)layers * n_slots * H * dk * dv * 4;
  const size_t es = elem_size(dtype);
  if (S_pool_new == S_pool) {
    if (!slot_out || slot_out == slot_in)
      return fail(KDA_ERR_ALIAS, "S_pool_new is S_pool: slot_out must name slots other than slot_in, "
                                 "or the committed states would be written");
  } else if (overlap(S_pool_new, pbytes, S_pool, pbytes)) {
    return fail(KDA_ERR_ALIAS, "S_pool_new partly overlaps S_pool");
  }
  if (overlap(out, heads * draft * dv * es, S_pool, pbytes) || overlap(out, heads * draft * dv * es, S_pool_new, pbytes))
    return fail(KDA_ERR_ALIAS, "out overlaps a state pool");
  kda::StepArgs a{};
  a.S_in = S_pool; a.S_out = S_pool_new;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out;
  a.n_accepted = n_accepted;
  a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.steps = draft; a.dtype = dtype; a.mode = mode;
  a.layers = layers; a.proj_steps = draft; a.ring_start = 0;
  a.out_head_stride = (int64_t)draft * dv; a.out_step_stride = dv;
  a.slot_in = slot_in; a.slot_out = slot_out ? slot_out : slot_in; a.n_slots = n_slots; a.layout = layout;
  return cuda_status(kda::launch_step(a, reinterpret_cast<cudaStream_t>(stream)), "kda_verify_replay_slots launch");
}

// ---------------------------------------------------------------------------
static int check_seqlens(const int32_t* cu, int n_seqs, int64_t T) {
  if (T < 0) return fail(KDA_ERR_SHAPE, "negative T");
  if (T > 0x7fffffffLL) return fail(KDA_ERR_SHAPE, "T=%lld exceeds 2^31-1 tokens", (long long)T);
  if (!cu) {
    if (n_seqs != 1) return fail(KDA_ERR_ARG, "cu_seqlens is NULL but n_seqs=%d (must be 1)", n_seqs);
    return KDA_OK;
  }
  if (n_seqs < 0) return fail(KDA_ERR_SHAPE, "negative n_seqs");
  if (cu[0] != 0) return fail(KDA_ERR_SHAPE, "cu_seqlens[0]=%d, must be 0", cu[0]);
  for (int n = 0; n < n_seqs; ++n)
    if (cu[n + 1] < cu[n]) return fail(KDA_ERR_SHAPE, "cu_seqlens decreases at %d", n);
  if (cu[n_seqs] != T) return fail(KDA_ERR_SHAPE, "cu_seqlens[n_seqs]=%d != T=%lld", cu[n_seqs], (long long)T);
  return KDA_OK;
}

int64_t kda_num_checkpoints(const int32_t* cu_seqlens, int n_seqs, int64_t T, int ckpt_stride) {
  if (ckpt_stride < 0) return fail(KDA_ERR_ARG, "negative ckpt_stride");
  if (int st = check_seqlens(cu_seqlens, n_seqs, T)) return st;
  ok();
  if (ckpt_stride == 0) return 0;
  if (!cu_seqlens) return T / ckpt_stride;
  int64_t n = 0;
  for (int i = 0; i < n_seqs; ++i) n += (cu_seqlens[i + 1] - cu_seqlens[i]) / ckpt_stride;
  return n;
}

// Per launch group of at most kMaxSeqs sequences: chunks of the group.
static int64_t group_chunks(const int32_t* cu, int N, int64_t T, int g0) {
  const int n = std::min(kda::kMaxSeqs, N - g0);
  int64_t c = 0;
  for (int i = g0; i < g0 + n; ++i) {
    const int64_t L = cu ? (int64_t)cu[i + 1] - cu[i] : T;
    c += (L + 63) / 64;
  }
  return c;
}

int64_t kda_prefill_workspace_bytes(const int32_t* cu_seqlens, int n_seqs, int64_t T, int H,
                                    int dk, int dv, int dtype) {
  if (int st = check_seqlens(cu_seqlens, n_seqs, T)) return st;
  if (H < 0) return fail(KDA_ERR_SHAPE, "negative H");
  ok();
  if (!kda::prefill_tc_supported(dk, dv, dtype)) return 0;
  const int N = cu_seqlens ? n_seqs : 1;
  int64_t worst = 0;
  for (int g0 = 0; g0 < N; g0 += kda::kMaxSeqs)
    worst = std::max(worst, group_chunks(cu_seqlens, N, T, g0));
  return worst * H * kda::prefill_tc_image_bytes(dv);
}

int kda_device_errors(int* flags) {
  if (!flags) return fail(KDA_ERR_ARG, "flags is NULL");
  int e = kda::read_and_clear_device_errors(flags);
  if (e == 0) e = kda::read_and_clear_prologue_errors(flags);
  if (e == 0) e = kda::read_and_clear_simt_errors(flags);
  if (e == 0) e = kda::read_and_clear_scan_errors(flags);
  if (e != 0) return cuda_status((cudaError_t)e, "kda_device_errors");
  return ok();
}

int kda_set_prefill_chain_columns(int cols) {
  if (cols != 0 && cols != 32 && cols != 64) return fail(KDA_ERR_ARG, "cols must be 0, 32 or 64");
  kda::g_chain_columns.store(cols, std::memory_order_relaxed);
  return ok();
}

// Checks shared by the prefill entry points; *need gets the checkpoint count and
// *done is set when there is nothing to launch.
static int check_prefill(const float* S0, const void* q, const void* k, const void* v, const void* g,
                         const void* beta, const int32_t* cu_seqlens, int n_seqs, int64_t T, int H, int dk,
                         int dv, int dtype, int chunk, int ckpt_stride, const void* o, const float* S_final,
                         const void* page_pool, int64_t page_bytes, const int32_t* ckpt_page_ids,
                         int64_t num_ckpt, int mode, int64_t* need, bool* done) {
  *need = 0;
  *done = false;
  if (int st = check_common(dk, dv, dtype, mode)) return st;
  if (chunk != 64) return fail(KDA_ERR_ARG, "chunk=%d: the kernels use 64-token chunks", chunk);
  if (ckpt_stride < 0 || (ckpt_stride % chunk) != 0)
    return fail(KDA_ERR_ARG, "ckpt_stride=%d must be a non-negative multiple of chunk=%d", ckpt_stride, chunk);
  if (H < 0) return fail(KDA_ERR_SHAPE, "negative H");
  if (int st = check_seqlens(cu_seqlens, n_seqs, T)) return st;
  const int N = cu_seqlens ? n_seqs : 1;
  if (N == 0 || H == 0) {
    *done = true;
    return KDA_OK;
  }
  const size_t es = elem_size(dtype);
  const size_t state_bytes = (size_t)N * H * dk * dv * 4;
  if (!S_final) return fail(KDA_ERR_ARG, "S_final is NULL");
  if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return fail(KDA_ERR_ARG, "null projection or output pointer");
  if ((S0 && !aligned16(S0)) || !aligned16(S_final) || !aligned16(q) || !aligned16(k) ||
      !aligned16(v) || !aligned16(g) || !aligned16(o))
    return fail(KDA_ERR_ALIGN, "state, projection and output pointers must be 16-byte aligned");
  if (overlap(S_final, state_bytes, S0, state_bytes))
    return fail(KDA_ERR_ALIAS, "S_final overlaps S0: the starting checkpoint must not be written");
  const size_t obytes = (size_t)T * H * dv * es;
  const size_t kbytes = (size_t)T * H * dk * es;
  if (overlap(o, obytes, q, kbytes) || overlap(o, obytes, k, kbytes) || overlap(o, obytes, g, kbytes) ||
      overlap(o, obytes, v, obytes) || overlap(o, obytes, S0, state_bytes) ||
      overlap(o, obytes, S_final, state_bytes))
    return fail(KDA_ERR_ALIAS, "o overlaps an input or the final state");
  *need = kda_num_checkpoints(cu_seqlens, n_seqs, T, ckpt_stride);
  if (*need < 0) return (int)*need;
  if (*need > 0) {
    if (!page_pool || !ckpt_page_ids) return fail(KDA_ERR_ARG, "checkpoints requested but page_pool or ckpt_page_ids is NULL");
    if (num_ckpt < *need)
      return fail(KDA_ERR_SHAPE, "num_ckpt=%lld < %lld checkpoints this prefill emits", (long long)num_ckpt,
                  (long long)*need);
    if (page_bytes < (int64_t)H * dk * dv * 4 || (page_bytes % 16) != 0)
      return fail(KDA_ERR_SHAPE, "page_bytes=%lld must be a multiple of 16 and >= H*dk*dv*4=%lld",
                  (long long)page_bytes, (long long)H * dk * dv * 4);
    if (!aligned16(page_pool)) return fail(KDA_ERR_ALIGN, "page_pool must be 16-byte aligned");
  }
  return KDA_OK;
}

int kda_prefill_chunked(const float* S0, const void* q, const void* k, const void* v,
                        const void* g, const void* beta, const int32_t* cu_seqlens, int n_seqs,
                        int64_t T, int H, int dk, int dv, int dtype, int chunk, int ckpt_stride,
                        void* o, float* S_final, void* page_pool, int64_t page_bytes,
                        const int32_t* ckpt_page_ids, int32_t* ckpt_pos, int64_t num_ckpt,
                        void* workspace, int64_t workspace_bytes,
                        int mode, kda_stream_t stream) {
  int64_t need = 0;
  bool done = false;
  if (int st = check_prefill(S0, q, k, v, g, beta, cu_seqlens, n_seqs, T, H, dk, dv, dtype, chunk, ckpt_stride, o,
                             S_final, page_pool, page_bytes, ckpt_page_ids, num_ckpt, mode, &need, &done))
    return st;
  if (done) return ok();
  const int N = cu_seqlens ? n_seqs : 1;
  if (workspace) {
    const int64_t ws_need = kda_prefill_workspace_bytes(cu_seqlens, n_seqs, T, H, dk, dv, dtype);
    if (ws_need < 0) return (int)ws_need;
    if (workspace_bytes < ws_need)
      return fail(KDA_ERR_SHAPE, "workspace_bytes=%lld < %lld needed", (long long)workspace_bytes,
                  (long long)ws_need);
    if (!aligned16(workspace)) return fail(KDA_ERR_ALIGN, "workspace must be 16-byte aligned");
    if (ws_need == 0) workspace = nullptr;
  }

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<int32_t> starts(N), lens(N), bases(N);
  int64_t cb = 0;
  for (int n = 0; n < N; ++n) {
    starts[n] = cu_seqlens ? cu_seqlens[n] : 0;
    lens[n] = cu_seqlens ? cu_seqlens[n + 1] - cu_seqlens[n] : (int32_t)T;
    bases[n] = (int32_t)cb;
    if (ckpt_stride > 0) cb += lens[n] / ckpt_stride;
  }
  // ~16 KB schedule block, passed to the kernel by value; kept off the stack
  static thread_local kda::PrefillSched sched_storage;
  kda::PrefillSched* sched = &sched_storage;
  int status = KDA_OK;
  for (int g0 = 0; g0 < N && status == KDA_OK; g0 += kda::kMaxSeqs) {
    const int n = std::min(kda::kMaxSeqs, N - g0);
    sched->n_seqs = n;
    std::vector<int32_t> idx(n);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int x, int y) { return lens[g0 + x] > lens[g0 + y]; });
    int max_len = 0;
    int32_t cbase = 0;
    for (int i = 0; i < n; ++i) {
      sched->order[i] = idx[i];
      sched->start[i] = starts[g0 + i];
      sched->len[i] = lens[g0 + i];
      sched->ckpt_base[i] = bases[g0 + i];
      sched->chunk_base[i] = cbase;
      sched->flags[i] = kda::kSeqEmit;
      sched->pos_base[i] = 0;
      cbase += (lens[g0 + i] + 63) / 64;
      max_len = std::max(max_len, lens[g0 + i]);
    }
    sched->chunk_base[n] = cbase;
    kda::PrefillArgs a{};
    const int64_t hs = (int64_t)H * dk * dv;
    a.S0 = S0 ? S0 + g0 * hs : nullptr;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.o = o;
    a.S_final = S_final + g0 * hs;
    a.page_pool = static_cast<char*>(page_pool);
    a.page_bytes = page_bytes;
    a.ckpt_page_ids = ckpt_page_ids;
    a.ckpt_pos = ckpt_pos;
    a.num_ckpt = need > 0 ? num_ckpt : 0;
    a.H = H; a.dk = dk; a.dv = dv; a.dtype = dtype; a.chunk = chunk;
    a.ckpt_stride = ckpt_stride; a.mode = mode;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.T = T;
    status = cuda_status(kda::launch_prefill(a, *sched, max_len, s), "kda_prefill_chunked launch");
  }
  return status;
}

// ---------------------------------------------------------------------------
static int scan_segments(int64_t T, int H, int dk, int dv, int ckpt_stride, int segments) {
  if (segments > 0) return segments;
  int dev = 0, n_sm = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) n_sm = v;
  }
  cudaGetLastError();                      // no device here: size for the GB300's 152 SMs
  return kda::prefill_scan_segments(T, H, dk, dv, ckpt_stride, n_sm);
}

int64_t kda_prefill_scan_workspace_bytes(int64_t T, int H, int dk, int dv, int dtype, int ckpt_stride, int segments) {
  if (int st = check_common(dk, dv, dtype, KDA_MODE_DECAY_FIRST)) return st;
  if (T < 0 || T > 0x7fffffffLL || H < 0) return fail(KDA_ERR_SHAPE, "T=%lld or H=%d out of range", (long long)T, H);
  if (ckpt_stride < 0 || ckpt_stride % 64 != 0) return fail(KDA_ERR_ARG, "ckpt_stride must be a multiple of 64");
  // (at most 1 + 254 * 3 pseudo-sequences in the first chain launch: within one launch group)
  if (segments < 0 || segments > 256) return fail(KDA_ERR_ARG, "segments=%d outside [0, 256]", segments);
  if (!kda::prefill_tc_supported(dk, dv, dtype))
    return fail(KDA_ERR_SHAPE, "the sequence-parallel prefill runs the tensor-core kernels: bf16, dk=128, dv 64 or 128");
  ok();
  const int64_t images = (T + 63) / 64 * H * kda::prefill_tc_image_bytes(dv);
  const int P = scan_segments(T, H, dk, dv, ckpt_stride, segments);
  return (images + 255) / 256 * 256 + kda::prefill_scan_scratch_bytes(T, H, dk, dv, ckpt_stride, P);
}

int kda_prefill_scan(const float* S0, const void* q, const void* k, const void* v, const void* g, const void* beta,
                     int64_t T, int H, int dk, int dv, int dtype, int chunk, int ckpt_stride, void* o, float* S_final,
                     void* page_pool, int64_t page_bytes, const int32_t* ckpt_page_ids, int32_t* ckpt_pos,
                     int64_t num_ckpt, void* workspace, int64_t workspace_bytes, int segments, int mode,
                     kda_stream_t stream) {
  int64_t need = 0;
  bool done = false;
  if (int st = check_prefill(S0, q, k, v, g, beta, nullptr, 1, T, H, dk, dv, dtype, chunk, ckpt_stride, o, S_final,
                             page_pool, page_bytes, ckpt_page_ids, num_ckpt, mode, &need, &done))
    return st;
  if (done) return ok();
  const int64_t ws_need = kda_prefill_scan_workspace_bytes(T, H, dk, dv, dtype, ckpt_stride, segments);
  if (ws_need < 0) return (int)ws_need;
  if (!workspace || workspace_bytes < ws_need)
    return fail(KDA_ERR_SHAPE, "workspace_bytes=%lld < %lld needed (kda_prefill_scan_workspace_bytes)",
                (long long)workspace_bytes, (long long)ws_need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return fail(KDA_ERR_ALIGN, "workspace must be 256-byte aligned");
  if (T == 0) {
    if (S0) return cuda_status(cudaMemcpyAsync(S_final, S0, (size_t)H * dk * dv * 4, cudaMemcpyDeviceToDevice,
                                               reinterpret_cast<cudaStream_t>(stream)), "kda_prefill_scan copy");
    return cuda_status(cudaMemsetAsync(S_final, 0, (size_t)H * dk * dv * 4, reinterpret_cast<cudaStream_t>(stream)),
                       "kda_prefill_scan zero");
  }
  const int P = scan_segments(T, H, dk, dv, ckpt_stride, segments);
  const int64_t images = ((T + 63) / 64 * H * kda::prefill_tc_image_bytes(dv) + 255) / 256 * 256;
  kda::PrefillArgs a{};
  a.S0 = S0;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.o = o;
  a.S_final = S_final;
  a.page_pool = static_cast<char*>(page_pool);
  a.page_bytes = page_bytes;
  a.ckpt_page_ids = ckpt_page_ids;
  a.ckpt_pos = ckpt_pos;
  a.num_ckpt = need > 0 ? num_ckpt : 0;
  a.H = H; a.dk = dk; a.dv = dv; a.dtype = dtype; a.chunk = chunk;
  a.ckpt_stride = ckpt_stride; a.mode = mode;
  a.workspace = workspace; a.workspace_bytes = images;
  a.T = T;
  return cuda_status(kda::launch_prefill_tc_scan(a, T, P, static_cast<char*>(workspace) + images,
                                                 reinterpret_cast<cudaStream_t>(stream)),
                     "kda_prefill_scan launch");
}

// ---------------------------------------------------------------------------
int kda_input_prep(const void* mixed_qkv, const void* conv_weight, int w, const void* window_in, void* window_out,
                   const void* g_logits, const void* beta_logits, float g_min, int act, const int32_t* cu_seqlens,
                   int n_seqs, int64_t T, int H, int dk, int dv, int dtype, void* q, void* k, void* v, void* g,
                   void* beta, int ckpt_stride, void* conv_ckpt, int64_t num_ckpt, kda_stream_t stream) {
  if (int st = check_common(dk, dv, dtype, KDA_MODE_DECAY_FIRST)) return st;
  if (w < 2 || w > 8) return fail(KDA_ERR_SHAPE, "conv kernel size w=%d outside [2, 8]", w);
  if (act != KDA_ACT_NONE && act != KDA_ACT_SILU) return fail(KDA_ERR_ARG, "act=%d is not a KDA_ACT_*", act);
  if (!(g_min < 0.f)) return fail(KDA_ERR_ARG, "g_min=%g must be negative", (double)g_min);
  if (H < 0) return fail(KDA_ERR_SHAPE, "negative H");
  if (int st = check_seqlens(cu_seqlens, n_seqs, T)) return st;
  if (ckpt_stride < 0) return fail(KDA_ERR_ARG, "negative ckpt_stride");
  const int N = cu_seqlens ? n_seqs : 1;
  if (T == 0 || H == 0 || N == 0) return ok();
  if (!mixed_qkv || !conv_weight || !g_logits || !beta_logits || !q || !k || !v || !g || !beta)
    return fail(KDA_ERR_ARG, "null pointer argument");
  const void* al[] = {mixed_qkv, conv_weight, window_in, window_out, g_logits, beta_logits, q, k, v, g, beta, conv_ckpt};
  for (const void* ptr : al)
    if (ptr && !aligned16(ptr)) return fail(KDA_ERR_ALIGN, "pointers must be 16-byte aligned");
  const int64_t need = ckpt_stride > 0 ? kda_num_checkpoints(cu_seqlens, n_seqs, T, ckpt_stride) : 0;
  if (conv_ckpt && ckpt_stride == 0) return fail(KDA_ERR_ARG, "conv_ckpt given with ckpt_stride 0");
  if (conv_ckpt && num_ckpt < need)
    return fail(KDA_ERR_SHAPE, "num_ckpt=%lld < %lld conv checkpoints", (long long)num_ckpt, (long long)need);
  const size_t es = elem_size(dtype);
  const size_t C = (size_t)H * (2 * dk + dv);
  const void* ins[] = {mixed_qkv, conv_weight, window_in, g_logits, beta_logits};
  const size_t in_bytes[] = {T * C * es, C * w * es, (size_t)N * (w - 1) * C * es, (size_t)T * H * dk * es,
                             (size_t)T * H * es};
  const void* outs[] = {q, k, v, g, beta, window_out, conv_ckpt};
  const size_t out_bytes[] = {(size_t)T * H * dk * es, (size_t)T * H * dk * es, (size_t)T * H * dv * es,
                              (size_t)T * H * dk * es, (size_t)T * H * es, (size_t)N * (w - 1) * C * es,
                              (size_t)(conv_ckpt ? num_ckpt : 0) * (w - 1) * C * es};
  for (int i = 0; i < 7; ++i) {
    for (int j = 0; j < 5; ++j)
      if (overlap(outs[i], out_bytes[i], ins[j], in_bytes[j])) return fail(KDA_ERR_ALIAS, "an output overlaps an input");
    for (int j = 0; j < i; ++j)
      if (overlap(outs[i], out_bytes[i], outs[j], out_bytes[j])) return fail(KDA_ERR_ALIAS, "two outputs overlap");
  }
  static thread_local kda::ProSched sched_storage;
  kda::ProSched* sched = &sched_storage;
  kda::ProArgs a{};
  a.mixed = mixed_qkv; a.weight = conv_weight; a.g_logits = g_logits; a.beta_logits = beta_logits;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.conv_ckpt = conv_ckpt; a.num_ckpt = conv_ckpt ? num_ckpt : 0;
  a.H = H; a.dk = dk; a.dv = dv; a.w = w; a.dtype = dtype; a.act = act; a.ckpt_stride = ckpt_stride;
  a.g_min = g_min; a.eps = 1e-6f;
  a.T = T;
  int64_t ckb = 0;
  for (int g0 = 0; g0 < N; g0 += kda::kMaxSeqs) {
    const int n = std::min(kda::kMaxSeqs, N - g0);
    sched->n_seqs = n;
    int32_t tb = 0;
    for (int i = 0; i < n; ++i) {
      const int32_t st0 = cu_seqlens ? cu_seqlens[g0 + i] : 0;
      const int32_t L = cu_seqlens ? cu_seqlens[g0 + i + 1] - st0 : (int32_t)T;
      sched->start[i] = st0;
      sched->len[i] = L;
      sched->ckpt_base[i] = (int32_t)ckb;
      if (ckpt_stride > 0) ckb += L / ckpt_stride;
      sched->tile_base[i] = tb;
      tb += (L + kda::kPrologueTile - 1) / kda::kPrologueTile;
    }
    sched->tile_base[n] = tb;
    const size_t woff = (size_t)g0 * (w - 1) * C * es;
    a.window_in = window_in ? static_cast<const char*>(window_in) + woff : nullptr;
    a.window_out = window_out ? static_cast<char*>(window_out) + woff : nullptr;
    cudaError_t e = kda::launch_prologue(a, *sched, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e, "kda_input_prep launch");
    // an empty sequence has no tile: its window passes through unchanged
    if (window_out) {
      const size_t wb = (size_t)(w - 1) * C * es;
      for (int i = 0; i < n && e == cudaSuccess; ++i) {
        if (sched->len[i] != 0) continue;
        char* dst = static_cast<char*>(a.window_out) + i * wb;
        e = window_in ? cudaMemcpyAsync(dst, static_cast<const char*>(a.window_in) + i * wb, wb,
                                        cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream))
                      : cudaMemsetAsync(dst, 0, wb, reinterpret_cast<cudaStream_t>(stream));
      }
      if (e != cudaSuccess) return cuda_status(e, "kda_input_prep window copy");
    }
  }
  return ok();
}

// ---------------------------------------------------------------------------
static int check_pack(const float* S, int64_t stride_b, int64_t stride_h, const float* flat,
                      int B, int H, int dk, int dv) {
  if (B < 0 || H < 0) return fail(KDA_ERR_SHAPE, "negative B or H");
  if (!head_dim_ok(dk) || !head_dim_ok(dv)) return fail(KDA_ERR_SHAPE, "dk, dv must be 32, 64 or 128");
  if ((int64_t)B * H == 0) return KDA_OK;
  if (!S || !flat) return fail(KDA_ERR_ARG, "null pointer argument");
  if (!aligned16(S) || !aligned16(flat)) return fail(KDA_ERR_ALIGN, "pointers must be 16-byte aligned");
  if (stride_b < 0 || stride_h < 0 || (stride_b % 4) || (stride_h % 4))
    return fail(KDA_ERR_ALIGN, "strides must be non-negative multiples of 4 elements");
  return KDA_OK;
}

int kda_pack_heads(const float* S, int64_t stride_b, int64_t stride_h, float* flat,
                   int64_t flat_elems, int B, int H, int dk, int dv, kda_stream_t stream) {
  if (int st = check_pack(S, stride_b, stride_h, flat, B, H, dk, dv)) return st;
  const int64_t n = (int64_t)B * H * dk * dv;
  if (flat_elems < n) return fail(KDA_ERR_SHAPE, "flat_elems=%lld < B*H*dk*dv=%lld", (long long)flat_elems, (long long)n);
  if (n == 0 && flat_elems == 0) return ok();
  if (!flat) return fail(KDA_ERR_ARG, "null flat");
  return cuda_status(kda::launch_pack(S, stride_b, stride_h, flat, flat_elems, B, H, dk, dv,
                                      reinterpret_cast<cudaStream_t>(stream)), "kda_pack_heads launch");
}

int kda_unpack_heads(const float* flat, float* S, int64_t stride_b, int64_t stride_h, int B, int H,
                     int dk, int dv, kda_stream_t stream) {
  if (int st = check_pack(S, stride_b, stride_h, flat, B, H, dk, dv)) return st;
  if ((int64_t)B * H == 0) return ok();
  return cuda_status(kda::launch_unpack(flat, S, stride_b, stride_h, B, H, dk, dv,
                                        reinterpret_cast<cudaStream_t>(stream)), "kda_unpack_heads launch");
}

// ---------------------------------------------------------------------------
struct kda_page_pool {
  char* base;
  int64_t page_bytes;
  int64_t n_pages;
  std::vector<int8_t> kind;
  std::set<int32_t> free_ids;
};

int kda_pool_create(void* device_base, int64_t page_bytes, int64_t n_pages, kda_page_pool** pool_out) {
  if (!pool_out) return fail(KDA_ERR_ARG, "pool_out is NULL");
  *pool_out = nullptr;
  if (n_pages < 0 || n_pages > 0x7fffffffLL) return fail(KDA_ERR_SHAPE, "n_pages out of range");
  if (page_bytes <= 0 || (page_bytes % 16)) return fail(KDA_ERR_SHAPE, "page_bytes must be a positive multiple of 16");
  if (n_pages > 0 && !device_base) return fail(KDA_ERR_ARG, "device_base is NULL");
  if (!aligned16(device_base)) return fail(KDA_ERR_ALIGN, "device_base must be 16-byte aligned");
  kda_page_pool* p = new kda_page_pool;
  p->base = static_cast<char*>(device_base);
  p->page_bytes = page_bytes;
  p->n_pages = n_pages;
  p->kind.assign((size_t)n_pages, KDA_PAGE_FREE);
  for (int64_t i = 0; i < n_pages; ++i) p->free_ids.insert(p->free_ids.end(), (int32_t)i);
  *pool_out = p;
  return ok();
}

int kda_pool_destroy(kda_page_pool* pool) {
  delete pool;
  return ok();
}

int kda_pool_alloc(kda_page_pool* pool, int kind, int64_t n, int32_t* page_ids_out) {
  if (!pool) return fail(KDA_ERR_ARG, "pool is NULL");
  if (kind != KDA_PAGE_KDA_STATE && kind != KDA_PAGE_MLA_KV) return fail(KDA_ERR_ARG, "bad page kind %d", kind);
  if (n < 0) return fail(KDA_ERR_ARG, "negative n");
  if (n > 0 && !page_ids_out) return fail(KDA_ERR_ARG, "page_ids_out is NULL");
  if ((int64_t)pool->free_ids.size() < n)
    return fail(KDA_ERR_NOMEM, "pool has %zu free pages, %lld requested", pool->free_ids.size(), (long long)n);
  for (int64_t i = 0; i < n; ++i) {
    auto it = pool->free_ids.begin();
    page_ids_out[i] = *it;
    pool->kind[*it] = (int8_t)kind;
    pool->free_ids.erase(it);
  }
  return ok();
}

int kda_pool_free(kda_page_pool* pool, int64_t n, const int32_t* page_ids) {
  if (!pool) return fail(KDA_ERR_ARG, "pool is NULL");
  if (n < 0 || (n > 0 && !page_ids)) return fail(KDA_ERR_ARG, "bad page id list");
  std::set<int32_t> seen;
  for (int64_t i = 0; i < n; ++i) {
    const int32_t id = page_ids[i];
    if (id < 0 || id >= pool->n_pages || pool->kind[id] == KDA_PAGE_FREE || !seen.insert(id).second)
      return fail(KDA_ERR_ARG, "page %d is not an allocated page (or is listed twice)", id);
  }
  for (int64_t i = 0; i < n; ++i) {
    pool->kind[page_ids[i]] = KDA_PAGE_FREE;
    pool->free_ids.insert(page_ids[i]);
  }
  return ok();
}

int64_t kda_pool_num_free(const kda_page_pool* pool) {
  if (!pool) return fail(KDA_ERR_ARG, "pool is NULL");
  return (int64_t)pool->free_ids.size();
}

int kda_pool_page_kind(const kda_page_pool* pool, int32_t page_id) {
  if (!pool || page_id < 0 || page_id >= pool->n_pages) return fail(KDA_ERR_ARG, "bad pool or page id");
  return pool->kind[page_id];
}

void* kda_pool_page_ptr(const kda_page_pool* pool, int32_t page_id) {
  if (!pool || page_id < 0 || page_id >= pool->n_pages) {
    fail(KDA_ERR_ARG, "bad pool or page id");
    return nullptr;
  }
  return pool->base + (int64_t)page_id * pool->page_bytes;
}

void* kda_pool_base(const kda_page_pool* pool) { return pool ? pool->base : nullptr; }
int64_t kda_pool_page_bytes(const kda_page_pool* pool) { return pool ? pool->page_bytes : (int64_t)KDA_ERR_ARG; }

static int check_state_page(const kda_page_pool* pool, int32_t page_id, int B, int H, int dk, int dv) {
  if (!pool) return fail(KDA_ERR_ARG, "pool is NULL");
  if (page_id < 0 || page_id >= pool->n_pages) return fail(KDA_ERR_ARG, "page id %d out of range", page_id);
  if (pool->kind[page_id] != KDA_PAGE_KDA_STATE)
    return fail(KDA_ERR_ARG, "page %d is not an allocated KDA state page", page_id);
  if ((int64_t)B * H * dk * dv * 4 > pool->page_bytes)
    return fail(KDA_ERR_SHAPE, "state of %lld bytes does not fit a %lld-byte page",
                (long long)B * H * dk * dv * 4, (long long)pool->page_bytes);
  return KDA_OK;
}

int kda_store_kda(kda_page_pool* pool, int32_t page_id, const float* S, int64_t stride_b,
                  int64_t stride_h, int B, int H, int dk, int dv, kda_stream_t stream) {
  if (int st = check_state_page(pool, page_id, B, H, dk, dv)) return st;
  float* page = reinterpret_cast<float*>(pool->base + (int64_t)page_id * pool->page_bytes);
  return kda_pack_heads(S, stride_b, stride_h, page, pool->page_bytes / 4, B, H, dk, dv, stream);
}

int kda_load_kda(const kda_page_pool* pool, int32_t page_id, float* S, int64_t stride_b,
                 int64_t stride_h, int B, int H, int dk, int dv, kda_stream_t stream) {
  if (int st = check_state_page(pool, page_id, B, H, dk, dv)) return st;
  const float* page = reinterpret_cast<const float*>(pool->base + (int64_t)page_id * pool->page_bytes);
  return kda_unpack_heads(page, S, stride_b, stride_h, B, H, dk, dv, stream);
}

double kda_snapshot_cost_ratio(int H, int dk, int dv) {
  if (H <= 0 || dk <= 0 || dv <= 0) {
    fail(KDA_ERR_ARG, "sizes must be positive");
    return -1.0;
  }
  ok();
  const double snap = (double)H * dk * dv;
  const double proj = (double)H * (3.0 * dk + dv + 1.0);
  return snap / proj;
}

}  // extern "C"

namespace kda {
int validate_prefill(const float* S0, const void* q, const void* k, const void* v, const void* g, const void* beta,
                     const int32_t* cu_seqlens, int n_seqs, int64_t T, int H, int dk, int dv, int dtype, int chunk,
                     int ckpt_stride, const void* o, const float* S_final, const void* page_pool, int64_t page_bytes,
                     const int32_t* ckpt_page_ids, int64_t num_ckpt, int mode) {
  int64_t need = 0;
  bool done = false;
  return check_prefill(S0, q, k, v, g, beta, cu_seqlens, n_seqs, T, H, dk, dv, dtype, chunk, ckpt_stride, o, S_final,
                       page_pool, page_bytes, ckpt_page_ids, num_ckpt, mode, &need, &done);
}
}  // namespace kda

namespace kda {
int set_error(int status, const char* msg) { return fail(status, "%s", msg); }
}  // namespace kda

// Prefill dispatch: the tensor-core kernel takes bf16 projections where it
// supports the shape; everything else runs the fp32 CUDA-core kernel.
namespace kda {
cudaError_t launch_prefill(const PrefillArgs& a, const PrefillSched& sched, int max_len, cudaStream_t s) {
  (void)max_len;
  bool handled = false;
  cudaError_t e = launch_prefill_tc(a, sched, s, &handled);
  if (handled) return e;
  return launch_prefill_simt(a, sched, s);
}
}  // namespace kda
