// Internal launch interface between the C ABI (kda_abi.cpp) and the kernels.
// Everything here assumes arguments were validated by the ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// One or more steps of the token recurrence per (b, h) head with the state
// held on chip across steps.  Decode: steps = 1, S_in == S_out.  Replay:
// steps = draft, per-sequence step counts from n_accepted.
struct StepArgs {
  const float* S_in;
  float* S_out;
  const void *q, *k, *v, *g, *beta;
  void* out;
  const int32_t* n_accepted;   // device [B] or nullptr (all heads run `steps`)
  int B, H, dk, dv, steps, dtype, mode;
  int layers;                  // stacked layers (replay); states [layers][B][H], projections [layers][proj_steps][B][H]
  int proj_steps;              // steps stored per layer in the projection arrays (>= steps)
  int ring_start;              // step s reads stored step (ring_start + s) mod proj_steps
  int64_t out_head_stride;     // elements between heads in `out`
  int64_t out_step_stride;     // elements between steps in `out`
  const int32_t* slot_in;      // device [B] or nullptr: states are [layers][n_slots][H], row b reads slot slot_in[b]
  const int32_t* slot_out;     // device [B]: row b writes slot slot_out[b] (used when slot_in is set)
  int64_t n_slots;
  int layout;                  // KDA_LAYOUT_KV: state (dk, dv); KDA_LAYOUT_VK: state (dv, dk)
  // decode with the input prologue fused in (mixed == nullptr: q, k, v, g, beta given)
  const void* mixed;           // [B][H (2 dk + dv)] raw rows [q | k | v]
  void* conv_state;            // [rows][w - 1][H (2 dk + dv)], row b (or slot_in[b]); shifted in place
  const void* conv_w;          // [H (2 dk + dv)][w]
  const void *g_logits, *beta_logits;       // [B][H][dk], [B][H]
  void *q_out, *k_out, *v_out, *g_out, *beta_out;   // prepared projections [B][H][...] or nullptr
  int conv_size, act;
  float g_min, eps;
};
cudaError_t launch_step(const StepArgs& a, cudaStream_t s);
cudaError_t launch_step_kv_f32(const StepArgs& a, cudaStream_t s);
cudaError_t launch_step_kv_bf16(const StepArgs& a, cudaStream_t s);
cudaError_t launch_step_vk_f32(const StepArgs& a, cudaStream_t s);
cudaError_t launch_step_vk_bf16(const StepArgs& a, cudaStream_t s);

// Sequence schedule of one prefill launch, passed by value as a kernel
// parameter: at most kMaxSeqs sequences.
constexpr int kMaxSeqs = 1024;
struct PrefillSched {
  int32_t n_seqs;
  int32_t order[kMaxSeqs];       // launch slot -> sequence (longest first)
  int32_t start[kMaxSeqs];       // first token of each sequence (relative to `base_token`)
  int32_t len[kMaxSeqs];         // tokens of each sequence
  int32_t ckpt_base[kMaxSeqs];   // index of each sequence's first checkpoint
  int32_t chunk_base[kMaxSeqs + 1];  // index of each sequence's first 64-token chunk; [n_seqs] = total
  // tensor-core chain only: per (pseudo-)sequence flags and the position of its first
  // token within the sequence it is a segment of (added to checkpoint positions)
  uint8_t flags[kMaxSeqs];
  int32_t pos_base[kMaxSeqs];
};
constexpr uint8_t kSeqEmit = 1;      // write outputs and checkpoints
constexpr uint8_t kSeqNoU = 2;       // drop the beta U term: the homogeneous (transition) recurrence

struct PrefillArgs {
  const float* S0;               // [n,H,dk,dv] (already offset to this launch) or nullptr
  const void *q, *k, *v, *g, *beta;  // token-major, offset to this launch's first token
  void* o;
  float* S_final;                // offset to this launch's first sequence
  char* page_pool;
  int64_t page_bytes;
  const int32_t* ckpt_page_ids;  // offset to this launch's first checkpoint
  int32_t* ckpt_pos;             // same offset, or nullptr
  int64_t num_ckpt;              // entries available from the offset
  void* workspace;               // chunk images of the tensor-core path, or nullptr
  int64_t workspace_bytes;
  int64_t T;                     // tokens in q/k/v/g/beta (all launch groups)
  int H, dk, dv, dtype, chunk, ckpt_stride, mode;
};
cudaError_t launch_prefill(const PrefillArgs& a, const PrefillSched& sched, int max_len,
                           cudaStream_t s);

// Input prologue (kda_prologue.cu): ShortConv over mixed_qkv rows [q | k | v],
// activation, per-head L2Norm of q and k, gates from logits.  One launch covers
// at most kMaxSeqs sequences; tiles of kPrologueTile tokens never span two sequences.
constexpr int kPrologueTile = 16;
struct ProSched {
  int32_t n_seqs;
  int32_t start[kMaxSeqs];       // first token of each sequence (absolute row of mixed)
  int32_t len[kMaxSeqs];
  int32_t ckpt_base[kMaxSeqs];   // index of each sequence's first conv checkpoint
  int32_t tile_base[kMaxSeqs + 1];
};
struct ProArgs {
  const void* mixed;             // [T][C], C = H (2 dk + dv)
  const void* weight;            // [C][w]
  const void* window_in;         // [n_seqs][w - 1][C] (offset to this launch) or nullptr
  void* window_out;              // same shape or nullptr
  const void *g_logits, *beta_logits;   // [T][H][dk], [T][H]
  void *q, *k, *v, *g, *beta;    // [T][H][dk] x 2, [T][H][dv], [T][H][dk], [T][H]
  void* conv_ckpt;               // [num_ckpt][w - 1][C] or nullptr
  int64_t num_ckpt;
  int64_t T;                     // rows of mixed and of the logits
  int H, dk, dv, w, dtype, act, ckpt_stride;
  float g_min, eps;
};
cudaError_t launch_prologue(const ProArgs& a, const ProSched& sched, cudaStream_t s);
cudaError_t launch_prologue_f32(const ProArgs& a, const ProSched& sched, cudaStream_t s);
cudaError_t launch_prologue_bf16(const ProArgs& a, const ProSched& sched, cudaStream_t s);
// OR the prologue kernels' device error words into *flags and clear them.
int read_and_clear_prologue_errors(int* flags);
int read_and_clear_prologue_errors_f32(int* flags);
int read_and_clear_prologue_errors_bf16(int* flags);

// Tensor-core path (kda_prefill_tc.cu): shapes it takes and workspace bytes per
// (64-token chunk, head).
bool prefill_tc_supported(int dk, int dv, int dtype);
int64_t prefill_tc_image_bytes(int dv);
// The two tensor-core kernels separately: chunk images of every chunk of `sched`
// into a.workspace, then the chain over `sched`'s (pseudo-)sequences.
cudaError_t launch_prefill_tc_prep(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s);
cudaError_t launch_prefill_tc_chain(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s);
// State columns per chain CTA chosen by kda_set_prefill_chain_columns(): 0 (by
// grid size), 32 or 64.
int prefill_chain_columns();
// Sequence-parallel prefill of one sequence (kda_scan.cu): the sequence cut into
// about `segments` pieces of whole checkpoint strides (fewer than 3 runs the plain
// chain); scratch of prefill_scan_scratch_bytes() for the same arguments.
int prefill_scan_segments(int64_t len, int H, int dk, int dv, int ckpt_stride, int n_sm);
int64_t prefill_scan_scratch_bytes(int64_t len, int H, int dk, int dv, int ckpt_stride, int segments);
cudaError_t launch_prefill_tc_scan(const PrefillArgs& a, int64_t len, int segments, void* scratch, cudaStream_t s);
// Copy the device error word to *flags and clear it (synchronises the device).
int read_and_clear_device_errors(int* flags);
// OR the CUDA-core prefill kernel's error word into *flags and clear it.
int read_and_clear_simt_errors(int* flags);
// OR the sequence-parallel scan kernel's error word into *flags and clear it.
int read_and_clear_scan_errors(int* flags);
// Record a failure message for kda_last_error() and return `status`.
int set_error(int status, const char* msg);
// The host-side argument checks of kda_prefill_chunked (everything but the
// workspace): KDA_OK or the status (and message) that call would return.
int validate_prefill(const float* S0, const void* q, const void* k, const void* v, const void* g, const void* beta,
                     const int32_t* cu_seqlens, int n_seqs, int64_t T, int H, int dk, int dv, int dtype, int chunk,
                     int ckpt_stride, const void* o, const float* S_final, const void* page_pool, int64_t page_bytes,
                     const int32_t* ckpt_page_ids, int64_t num_ckpt, int mode);

// Flat <-> strided (B,H,dk,dv) copies.  pack zero-fills flat past B*H*dk*dv.
cudaError_t launch_pack(const float* S, int64_t stride_b, int64_t stride_h, float* flat,
                        int64_t flat_elems, int B, int H, int dk, int dv, cudaStream_t s);
cudaError_t launch_unpack(const float* flat, float* S, int64_t stride_b, int64_t stride_h,
                          int B, int H, int dk, int dv, cudaStream_t s);

}  // namespace kda
