/*
 * kda.h -- C ABI of the GB300 (sm_103a) KDA gated delta-rule library.
 *
 * The operations follow two pages:
 *   [SERVE] "【轻量化复刻大模型 / KIMI K3】Serve 模块交互式演示"
 *           (www.cveoy.top/t/topic/qHUG): §1.1 projection cache and
 *           snapshot_cost_ratio, §1.2 verify_and_replay, §1.3 the KDA
 *           recurrence (kda_step), §1.5 the unified page pool and
 *           pack_heads / unpack_heads, Tab 7 store_kda / load_kda.
 *   [CACHE] "Kimi Linear 的 KDA 缓存：SGLang、vLLM 与 Mooncake Store 全链路"
 *           (imreese.github.io/blogs/kimi-kda-cache-sglang-vllm-mooncake-store):
 *           "KDA 的递推与充分状态" (decay first, per-key-channel gates),
 *           "预填充为什么能分块并行" (chunked WY/UT form, chunk 64),
 *           "SGLang：从一次较长的 extend 调用中提取检查点" (chunk-aligned
 *           intermediate states), "检查点状态池的内存成本" (FP32 state).
 *
 * Conventions (all entry points):
 *  - Every call returns an int status: KDA_OK (0) or a negative KDA_ERR_*.
 *    Arguments are validated on the host before anything is launched; a call
 *    that fails validation launches nothing and writes nothing.
 *    kda_last_error() gives a message for the calling thread's last failure.
 *  - The caller owns all memory. No entry point allocates device memory.
 *  - Pointers named "device" must be device (or managed) memory of the
 *    current device; "host" pointers are plain host memory.
 *  - Launches are asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream). Device-side errors surface on later syncs.
 *  - State tensors are fp32, layout (..., dk, dv) row-major: key channels are
 *    rows, dv is contiguous. Projections q, k, g are (..., dk), v is
 *    (..., dv), beta is (...) -- all of one dtype `dtype` (KDA_F32 or
 *    KDA_BF16). Outputs o take the same dtype as the projections.
 *  - Supported head sizes: dk, dv in {32, 64, 128}.
 *  - Base pointers of state and projection arrays must be 16-byte aligned.
 *  - Gates g are per-key-channel log-decays in [g_min, 0] with g_min >= -10
 *    (the pages draw g = g_min * sigmoid(.), g_min = -5); beta in [0, 1].
 *
 * Modes: KDA_MODE_DECAY_FIRST ([CACHE]: S' = Diag(e^g) S; delta = v - S'^T k;
 * S = S' + beta k delta^T; o = S^T q) and KDA_MODE_UNDECAYED_DELTA ([SERVE]
 * §1.3: delta = v - S^T k taken against the undecayed state;
 * S = Diag(e^g) S + beta k delta^T; o = S^T q).
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define KDA_OK          0
#define KDA_ERR_ARG    -1   /* null pointer, bad enum, bad scalar argument   */
#define KDA_ERR_SHAPE  -2   /* unsupported or inconsistent sizes             */
#define KDA_ERR_DTYPE  -3   /* unsupported dtype                             */
#define KDA_ERR_ALIGN  -4   /* pointer not aligned as required               */
#define KDA_ERR_CUDA   -5   /* a CUDA runtime call failed                    */
#define KDA_ERR_NOMEM  -6   /* page pool exhausted                           */
#define KDA_ERR_ALIAS  -7   /* an output overlaps an input it must not touch */

/* dtypes of projections / outputs */
#define KDA_F32   0
#define KDA_BF16  1

/* orderings of the recurrence */
#define KDA_MODE_DECAY_FIRST      0
#define KDA_MODE_UNDECAYED_DELTA  1

/* activations of the input prologue */
#define KDA_ACT_NONE  0
#define KDA_ACT_SILU  1

/* page kinds of the unified pool ([SERVE] §1.5: one free list, two kinds) */
#define KDA_PAGE_FREE       0
#define KDA_PAGE_KDA_STATE  1
#define KDA_PAGE_MLA_KV     2

/* limits */
#define KDA_MAX_DRAFT            16    /* replay steps per call                */
#define KDA_MAX_SEQS_PER_LAUNCH  1024  /* prefill splits larger batches        */

typedef struct CUstream_st* kda_stream_t;   /* identical to cudaStream_t */

int         kda_version(void);
const char* kda_status_string(int status);
const char* kda_last_error(void);

/*
 * kda_decode_step -- one token of the recurrence for B*H heads, in place.
 * [SERVE] §1.3 kda_step; [CACHE] "KDA 的递推与充分状态".
 *   S     device fp32 [B,H,dk,dv]    in/out, updated in place
 *   q,k,g device dtype [B,H,dk]      in
 *   v     device dtype [B,H,dv]      in
 *   beta  device dtype [B,H]         in
 *   o     device dtype [B,H,dv]      out: o = S_new^T q
 * B == 0 or H == 0 is a no-op. o must not overlap S.
 */
int kda_decode_step(float* S, const void* q, const void* k, const void* v,
                    const void* g, const void* beta, void* o,
                    int B, int H, int dk, int dv, int dtype, int mode,
                    kda_stream_t stream);

/*
 * kda_verify_replay -- clone the committed state and replay the accepted
 * prefix of a draft. [SERVE] §1.2 verify_and_replay, Tab 3 §6.4.
 *   S_committed  device fp32 [B,H,dk,dv]        in, never written
 *   q,k,g        device dtype [draft,B,H,dk]    in (draft-projection cache layout)
 *   v            device dtype [draft,B,H,dv]    in
 *   beta         device dtype [draft,B,H]       in
 *   n_accepted   device int32 [B]               in; clamped to [0, draft]
 *   S_new        device fp32 [B,H,dk,dv]        out: state after n_b steps
 *   out          device dtype [B,H,draft,dv]    out: step outputs, zero for
 *                                               steps >= n_b
 * 1 <= draft <= KDA_MAX_DRAFT. S_new must not overlap S_committed
 * (KDA_ERR_ALIAS): the committed state is shared and must stay intact.
 */
int kda_verify_replay(const float* S_committed, const void* q, const void* k,
                      const void* v, const void* g, const void* beta,
                      const int32_t* n_accepted, float* S_new, void* out,
                      int draft, int B, int H, int dk, int dv, int dtype, int mode,
                      kda_stream_t stream);

/*
 * kda_verify_replay_layers -- kda_verify_replay for the KDA layers of one model
 * in a single launch: every layer replays the same accepted prefix of its own
 * draft projections from its own committed state.  [SERVE] §1.2 (one
 * verify_and_replay per KDA layer; the accepted count is per sequence, shared
 * by the layers).  kda_verify_replay is the case layers = 1.
 *   S_committed  device fp32 [layers,B,H,dk,dv]       in, never written
 *   q,k,g        device dtype [layers,draft,B,H,dk]   in (each layer in the
 *                                                      draft-projection cache layout)
 *   v            device dtype [layers,draft,B,H,dv]   in
 *   beta         device dtype [layers,draft,B,H]      in
 *   n_accepted   device int32 [B]                     in; clamped to [0, draft]
 *   S_new        device fp32 [layers,B,H,dk,dv]       out
 *   out          device dtype [layers,B,H,draft,dv]   out, zero for steps >= n_b
 * Same rules and errors as kda_verify_replay; layers = 0 (or B*H = 0) is a no-op.
 */
int kda_verify_replay_layers(int layers, const float* S_committed, const void* q,
                             const void* k, const void* v, const void* g,
                             const void* beta, const int32_t* n_accepted, float* S_new,
                             void* out, int draft, int B, int H, int dk, int dv,
                             int dtype, int mode, kda_stream_t stream);

/* state layouts of the slot-pool entry points */
#define KDA_LAYOUT_KV  0   /* state (dk, dv): key channels are rows, dv contiguous   */
#define KDA_LAYOUT_VK  1   /* state (dv, dk): value channels are rows, dk contiguous */

/*
 * kda_decode_step_slots -- kda_decode_step on states kept in a slot pool, in
 * either layout: one layer of a serving engine's recurrent-state buffer,
 * [slots, heads, d_v, d_k] for KDA_LAYOUT_VK.  [CACHE] "先统一记号：矩阵状态不等于
 * 完整检查点" (the state is written [local_heads, d_k, d_v]; kernels and state
 * pools may store it transposed, [local_heads, d_v, d_k]) and "一个逻辑检查点如何
 * 展开" (SGLang's buffer [num_kda_layers, slots, local_heads, d_v, d_k]: one
 * slot spans every KDA layer).  Same recurrence as kda_decode_step.
 *   S_pool    device fp32 [n_slots,H,dk,dv] (KDA_LAYOUT_KV) or
 *             [n_slots,H,dv,dk] (KDA_LAYOUT_VK), updated in place; for layer l
 *             of a [layers,n_slots,H,...] buffer pass its base + l*n_slots*H*dk*dv
 *   slot_ids  device int32 [B]: batch row b updates slot slot_ids[b].  An id
 *             outside [0, n_slots) (such as -1 for a padded row) touches no
 *             state and gives a zero output row.  Valid ids must be distinct
 *             (two rows on one slot race); device memory, so not checked.
 *   q,k,g,v,beta,o  as kda_decode_step ([B,H,...]); o must not overlap S_pool
 * Errors: as kda_decode_step; KDA_ERR_ARG for a bad layout or NULL slot_ids,
 * KDA_ERR_SHAPE for n_slots < 1.
 */
int kda_decode_step_slots(float* S_pool, int64_t n_slots, const int32_t* slot_ids, int layout,
                          const void* q, const void* k, const void* v, const void* g,
                          const void* beta, void* o, int B, int H, int dk, int dv, int dtype,
                          int mode, kda_stream_t stream);

/*
 * kda_decode_step_fused -- one decode token with the input prologue of
 * kda_input_prep fused in: the raw mixed_qkv row of each sequence passes
 * through the causal ShortConv (its window shifted in place), the activation,
 * per-head L2Norm of q and k and the gates from their logits, then one step of
 * the recurrence, in one launch.  [CACHE] "KDA 的递推与充分状态" (the prologue
 * and the recurrence), "一个逻辑检查点如何展开" (SGLang keeps the conv window
 * [layers, slots, kernel_size - 1, qkv_width] beside the recurrent state);
 * [SERVE] §1.3.  Same readings of the prologue as kda_input_prep.
 *   S          device fp32: [B,H,<state>] (slot_ids NULL) or a pool
 *              [n_slots,H,<state>]; <state> per layout as in the slot entry points
 *   slot_ids   device int32 [B] or NULL: row b uses slot slot_ids[b] of S and of
 *              conv_state; ids outside [0, n_slots) give zero output and touch
 *              nothing; valid ids must be distinct
 *   conv_state device dtype [B or n_slots, w-1, C], C = H*(2*dk + dv), in/out
 *   mixed_qkv  device dtype [B, C] in; conv_weight [C, w] in, 2 <= w <= 4 (the
 *              window sits in registers; kda_input_prep takes up to 8)
 *   g_logits   device dtype [B, H, dk]; beta_logits [B, H]   in
 *   o          device dtype [B, H, dv] out
 *   q_out, k_out, g_out [B,H,dk], v_out [B,H,dv], beta_out [B,H]: all NULL, or
 *              all given to receive the prepared projections (for a
 *              draft-projection cache); rows of skipped ids are left unwritten
 * Errors: as kda_decode_step and kda_input_prep; KDA_ERR_ALIAS when any two
 * arguments overlap.
 */
int kda_decode_step_fused(float* S, int64_t n_slots, const int32_t* slot_ids, int layout,
                          void* conv_state, const void* mixed_qkv, const void* conv_weight, int w,
                          const void* g_logits, const void* beta_logits, float g_min, int act,
                          void* o, void* q_out, void* k_out, void* v_out, void* g_out, void* beta_out,
                          int B, int H, int dk, int dv, int dtype, int mode, kda_stream_t stream);

/*
 * kda_verify_replay_slots -- kda_verify_replay_layers on states kept in slot
 * pools, in either layout.  Row b of layer l replays the accepted prefix from
 * slot slot_in[b] of layer l of S_pool and writes the resulting state into
 * slot slot_out[b] of layer l of S_pool_new.  [SERVE] §1.2 verify_and_replay
 * over the [CACHE] "一个逻辑检查点如何展开" slot buffer.
 *   S_pool      device fp32 [layers,n_slots,H,<state>]  in, the committed states
 *   S_pool_new  device fp32 [layers,n_slots,H,<state>]  out.  It may be S_pool
 *               itself (states move between slots, a commit is then a change of
 *               slot ids): slot_out must then be given, its valid ids distinct
 *               and disjoint from every valid slot_in id so that no committed
 *               state is written -- device memory, so not checked
 *   slot_in     device int32 [B]
 *   slot_out    device int32 [B], or NULL for slot_in (needs S_pool_new != S_pool)
 *   q,k,g,v,beta,n_accepted,out  as kda_verify_replay_layers
 * <state> is (dk,dv) for KDA_LAYOUT_KV, (dv,dk) for KDA_LAYOUT_VK.  A row
 * whose slot_in or slot_out id is outside [0, n_slots) touches no state and
 * gives zero output rows.
 * Errors: as kda_verify_replay_layers; KDA_ERR_ALIAS when S_pool_new is S_pool
 * without a distinct slot_out array, or partly overlaps it.
 */
int kda_verify_replay_slots(int layers, const float* S_pool, float* S_pool_new, int64_t n_slots,
                            const int32_t* slot_in, const int32_t* slot_out, int layout,
                            const void* q, const void* k, const void* v, const void* g,
                            const void* beta, const int32_t* n_accepted, void* out,
                            int draft, int B, int H, int dk, int dv, int dtype, int mode,
                            kda_stream_t stream);

/*
 * Raw-input ring -- the window of raw draft projections that a commit replays
 * ([SERVE] Tab 4 §7.2, RawInputRing / fold-every-commit: during verification
 * each draft step's raw (q, k, v, g, beta) is streamed into a per-slot window
 * instead of snapshotting the state; once the window holds `capacity` steps
 * a push overwrites the oldest; a commit replays the accepted prefix).
 * The ring lives in device memory the caller provides (kda_ring_bytes bytes,
 * 256-byte aligned) and is laid out like the draft-projection cache
 * ([capacity][B][H][D] per tensor), so kda_verify_replay_ring reads it in
 * place.  The handle is host state (the push count); one thread at a time.
 *   kda_ring_bytes    device bytes of a ring (negative KDA_ERR_* if invalid):
 *                     1 <= capacity <= KDA_MAX_DRAFT, dk, dv in {32,64,128}
 *   kda_ring_create   wrap device_base; the window starts empty
 *   kda_ring_push     copy one step (device q,k,g [B,H,dk], v [B,H,dv],
 *                     beta [B,H], dtype of the ring) in, asynchronously on stream
 *   kda_ring_len      steps in the window (<= capacity)
 *   kda_ring_window   copy the window out, oldest first, as [len,B,H,D]
 *   kda_ring_reset    empty the window (after a commit)
 *   kda_verify_replay_ring  kda_verify_replay over the window: S_committed
 *                     [B,H,dk,dv] fp32 never written, n_accepted [B] clamped to
 *                     [0, len], S_new [B,H,dk,dv], out [B,H,len,dv]
 */
typedef struct kda_raw_ring kda_raw_ring;
int64_t kda_ring_bytes(int capacity, int B, int H, int dk, int dv, int dtype);
int kda_ring_create(void* device_base, int capacity, int B, int H, int dk, int dv,
                    int dtype, kda_raw_ring** ring_out);
int kda_ring_destroy(kda_raw_ring* ring);
int kda_ring_reset(kda_raw_ring* ring);
int kda_ring_len(const kda_raw_ring* ring);
int kda_ring_push(kda_raw_ring* ring, const void* q, const void* k, const void* v,
                  const void* g, const void* beta, kda_stream_t stream);
int kda_ring_window(const kda_raw_ring* ring, void* q, void* k, void* v, void* g,
                    void* beta, kda_stream_t stream);
int kda_verify_replay_ring(const kda_raw_ring* ring, const float* S_committed,
                           const int32_t* n_accepted, float* S_new, void* out, int mode,
                           kda_stream_t stream);

/*
 * kda_num_checkpoints -- number of checkpoint states a prefill will emit:
 * sum over sequences of floor(L_n / ckpt_stride). Host only.
 *   cu_seqlens  host int32 [n_seqs+1] or NULL (one sequence of T tokens)
 * Returns the count (>= 0) or a negative KDA_ERR_*.
 */
int64_t kda_num_checkpoints(const int32_t* cu_seqlens, int n_seqs, int64_t T,
                            int ckpt_stride);

/*
 * kda_prefill_chunked -- chunked (WY/UT) prefill of packed sequences with
 * chunk-aligned checkpoint emission. [CACHE] "预填充为什么能分块并行",
 * "SGLang：从一次较长的 extend 调用中提取检查点"; [SERVE] §1.5, Tab 7.
 *   S0          device fp32 [n_seqs,H,dk,dv] in, never written; NULL = zero state
 *   q,k,g       device dtype [T,H,dk]        in (token-major, packed sequences)
 *   v           device dtype [T,H,dv]        in
 *   beta        device dtype [T,H]           in
 *   cu_seqlens  host int32 [n_seqs+1]        sequence boundaries, cu[0] = 0,
 *                                            non-decreasing, cu[n_seqs] = T;
 *                                            NULL means one sequence (n_seqs = 1)
 *   chunk       must be 64
 *   ckpt_stride multiple of chunk, or 0 for no checkpoints
 *   o           device dtype [T,H,dv]        out
 *   S_final     device fp32 [n_seqs,H,dk,dv] out, must not overlap S0
 *   page_pool   device base of the page arena (required if checkpoints > 0)
 *   page_bytes  bytes per page, multiple of 16, >= H*dk*dv*4
 *   ckpt_page_ids device int32 [num_ckpt]    page index of checkpoint c
 *   ckpt_pos    device int32 [num_ckpt] out  boundary position of checkpoint c
 *                                            within its sequence (may be NULL)
 *   num_ckpt    entries in ckpt_page_ids; must be >= kda_num_checkpoints()
 *   workspace   device scratch for the tensor-core kernels, or NULL;
 *   workspace_bytes  its size, >= kda_prefill_workspace_bytes() when used
 * Checkpoint c (sequence-major, then position) is the state after the first
 * j*ckpt_stride tokens of its sequence, j >= 1, written into page
 * ckpt_page_ids[c] in pack_heads layout ([1,H,dk,dv] flat) with the rest of
 * the page zeroed. Positions count from each sequence's first token.
 * Page ids must index pages inside the arena (not checked: device memory).
 * Kernels: bf16 projections with dk = 128 and dv in {64, 128} run on tcgen05
 * tensor cores (bf16 operands, fp32 accumulation and state) when a workspace
 * is given; every other case, and a NULL workspace, runs the fp32 CUDA-core
 * kernel. Both take g in [-10, 0]: a gate outside that range (or NaN) is not
 * rejected on the host (it is device data) but raises KDA_DEVERR_GATE in
 * kda_device_errors(), and the call's results are then not to be trusted. The workspace is only touched during the call's kernels (stream
 * order); calls sharing one workspace must be ordered on one stream.
 */
int kda_prefill_chunked(const float* S0, const void* q, const void* k,
                        const void* v, const void* g, const void* beta,
                        const int32_t* cu_seqlens, int n_seqs, int64_t T,
                        int H, int dk, int dv, int dtype, int chunk, int ckpt_stride,
                        void* o, float* S_final,
                        void* page_pool, int64_t page_bytes,
                        const int32_t* ckpt_page_ids, int32_t* ckpt_pos, int64_t num_ckpt,
                        void* workspace, int64_t workspace_bytes,
                        int mode, kda_stream_t stream);

/*
 * kda_prefill_scan -- kda_prefill_chunked for one long sequence, sequence-parallel
 * inside the GPU (the context-parallel prefix scan: [CACHE] "预填充为什么能分块并行",
 * every token transition is a diagonal matrix minus a rank-one matrix, so the
 * state after a segment is affine in the state before it, S_end = M S_start + L;
 * [SERVE] §1.7, KCP passes one state per rank whatever the length).  The sequence
 * is cut into about `segments` pieces of whole checkpoint strides (whole 64-token
 * chunks without checkpoints); the chunk images are built once; one chain launch
 * runs the first piece from S0 and, for each middle piece, its state from zero and
 * its transition (dk/dv pseudo-sequences from identity columns with the beta U
 * term dropped); an fp32 scan gives every piece's start state; a second chain
 * launch runs the pieces from their starts with outputs and checkpoints.  Worth
 * it when H * dv / 64 chains leave most SMs idle (few heads, long sequence);
 * results match kda_prefill_chunked within the bf16 tolerances, not bitwise.
 *   Arguments as kda_prefill_chunked for one sequence (no cu_seqlens), plus
 *   segments   0 = choose: the most pieces whose first chain launch fits one CTA
 *              per SM; 1 or 2 = the plain chain; at most 256; the count is
 *              rounded so pieces are whole strides
 *   workspace  device, 256-byte aligned, >= kda_prefill_scan_workspace_bytes(...)
 *              for the same T, H, dk, dv, dtype, ckpt_stride, segments
 * Tensor-core shapes only (bf16, dk = 128, dv in {64, 128}): others KDA_ERR_SHAPE.
 */
int kda_prefill_scan(const float* S0, const void* q, const void* k, const void* v,
                     const void* g, const void* beta, int64_t T, int H, int dk, int dv,
                     int dtype, int chunk, int ckpt_stride, void* o, float* S_final,
                     void* page_pool, int64_t page_bytes, const int32_t* ckpt_page_ids,
                     int32_t* ckpt_pos, int64_t num_ckpt, void* workspace,
                     int64_t workspace_bytes, int segments, int mode, kda_stream_t stream);
int64_t kda_prefill_scan_workspace_bytes(int64_t T, int H, int dk, int dv, int dtype,
                                         int ckpt_stride, int segments);

/*
 * kda_prefill_workspace_bytes -- device scratch the tensor-core prefill needs
 * for these sequences (0 when the shape runs on the CUDA-core kernel). The
 * scratch holds, per 64-token chunk and head, the chunk's WY/UT operands in
 * tensor-core layout. Host only; same sequence arguments as the prefill.
 * Returns the byte count (>= 0) or a negative KDA_ERR_*.
 */
int64_t kda_prefill_workspace_bytes(const int32_t* cu_seqlens, int n_seqs, int64_t T,
                                    int H, int dk, int dv, int dtype);

/*
 * kda_device_errors -- read and clear the library's device error word.
 * Bit 0 (KDA_DEVERR_WAIT): a kernel gave up waiting on an mbarrier (about
 * one second) and returned early, so that call's outputs are invalid.
 * Bit 1 (KDA_DEVERR_GATE): a chunked prefill (kda_prefill_chunked and the
 * calls built on it) read a gate g outside [-10, 0] or a NaN gate. Its
 * kernels split each pairwise decay at a reference token per 16-token block,
 * so a factor can reach e^(8 |g|): finite for g >= -10, not beyond. The
 * call's outputs may then hold inf or NaN. ([SERVE] §1.3 draws
 * g = g_min sigmoid(.) in [g_min, 0]; the pages use g_min = -5.)
 * Synchronises the device. *flags receives the word; returns KDA_OK or
 * KDA_ERR_CUDA.
 */
#define KDA_DEVERR_WAIT  1
#define KDA_DEVERR_GATE  2
int kda_device_errors(int* flags);

/*
 * kda_set_prefill_chain_columns -- a tuning knob of the tensor-core prefill
 * (kda_prefill_chunked, kda_prefill_scan and the variants built on them):
 * how many columns of each head's state one CTA of the sequential chunk
 * chain owns ([CACHE] "预填充为什么能分块并行": the chunks of a sequence
 * are walked in order; the dv columns of the state evolve independently).
 *   cols  32 or 64; 0 (the default) chooses per call: 32 while twice the
 *         number of 64-column CTAs still fits the device's SMs, else 64.
 * Results agree to rounding either way. Process-wide; applies to calls
 * issued after it returns. Errors: KDA_ERR_ARG for any other value (the
 * setting is left as it was).
 */
int kda_set_prefill_chain_columns(int cols);

/*
 * kda_prefill_chunked_noalloc -- kda_prefill_chunked without a caller
 * workspace. It allocates no device memory, for callers that cannot call
 * cudaMalloc/cudaFree at call time: serving loops that forbid them because
 * they synchronise the whole device and stall every stream, and code embedded
 * in a host framework that owns all device memory through its own allocator.
 * (The pages have no counterpart: this is an interface for such callers.)
 * Same arguments, layouts and results as kda_prefill_chunked. The
 * tensor-core scratch comes from one fixed array of
 * KDA_NOALLOC_SCRATCH_BYTES in device memory, which every GPU that loads the
 * library holds until the process exits; a call whose shape needs more
 * (kda_prefill_workspace_bytes() larger than that) fails with KDA_ERR_SHAPE
 * and launches nothing. Shapes that need no scratch run the fp32 CUDA-core
 * kernel as kda_prefill_chunked does with a NULL workspace.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * The address is kept per device ordinal for the life of the process: it
 * assumes the runtime's primary context on each device, with no
 * cudaDeviceReset in between (after a reset, or under a context the caller
 * created through the driver API, the kept address would be stale).
 * All calls share the one array: calls whose kernels overlap on the GPU (on
 * different streams, or from different threads) race on it and must be
 * ordered by the caller. Nothing in it needs clearing between calls: every
 * byte a call reads was written earlier in the same call.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64ull << 20)   /* 64 MiB */
int kda_prefill_chunked_noalloc(const float* S0, const void* q, const void* k,
                                const void* v, const void* g, const void* beta,
                                const int32_t* cu_seqlens, int n_seqs, int64_t T,
                                int H, int dk, int dv, int dtype, int chunk, int ckpt_stride,
                                void* o, float* S_final,
                                void* page_pool, int64_t page_bytes,
                                const int32_t* ckpt_page_ids, int32_t* ckpt_pos, int64_t num_ckpt,
                                int mode, kda_stream_t stream);

/*
 * kda_prefill_chunked_host -- kda_prefill_chunked with the projections, S0,
 * o and S_final in host memory: the call moves them itself, cut into
 * segments of at most `segment_tokens` tokens so that the copies of one
 * segment overlap the computation of its neighbours (two internal copy
 * streams, events, the compute on `stream`).  A sequence is cut only at a
 * multiple of ckpt_stride (of 64 without checkpoints) from its own start, so
 * the results are the same bits as kda_prefill_chunked on device copies.
 * [CACHE] "预填充为什么能分块并行"; the pages run prefill from device memory.
 *   S0, q, k, v, g, beta   host, same shapes as kda_prefill_chunked (S0 may be
 *                          NULL = zero state); pinned (page-locked) memory
 *                          is needed for the copies to overlap
 *   o, S_final             host outputs, same shapes
 *   page_pool, ckpt_page_ids, ckpt_pos   device, as in kda_prefill_chunked;
 *                          ckpt_pos (optional) gets positions from each
 *                          sequence's start
 *   scratch                device, 256-byte aligned, at least
 *                          kda_prefill_host_scratch_bytes(...) bytes; owned by
 *                          the caller, busy until `stream` passes this call
 * Returns when everything is enqueued; all copies and kernels are ordered
 * before later work on `stream` (synchronise it before reading o, S_final).
 * Errors: as kda_prefill_chunked, KDA_ERR_SHAPE for a small scratch,
 * KDA_ERR_ALIGN for an unaligned scratch, KDA_ERR_CUDA for a failed copy.
 */
int64_t kda_prefill_host_scratch_bytes(int H, int dk, int dv, int dtype, int ckpt_stride,
                                       int64_t segment_tokens);
int kda_prefill_chunked_host(const float* S0, const void* q, const void* k, const void* v,
                             const void* g, const void* beta, const int32_t* cu_seqlens,
                             int n_seqs, int64_t T, int H, int dk, int dv, int dtype,
                             int chunk, int ckpt_stride, void* o, float* S_final,
                             void* page_pool, int64_t page_bytes,
                             const int32_t* ckpt_page_ids, int32_t* ckpt_pos,
                             int64_t num_ckpt, void* scratch, int64_t scratch_bytes,
                             int64_t segment_tokens, int mode, kda_stream_t stream);

/*
 * kda_input_prep -- the input prologue of a KDA layer for prefill: causal
 * depthwise ShortConv over the rows of mixed_qkv, activation, per-head L2Norm of
 * q and k, and the gates from their logits, writing the q, k, v, g, beta that
 * kda_prefill_chunked reads.  [CACHE] "KDA 的递推与充分状态" (projection, causal
 * short convolution and activation, L2Norm of Q and K), "先统一记号：矩阵状态不等于
 * 完整检查点" (the ShortConv window: the kernel_size - 1 most recent inputs),
 * "SGLang：从一次较长的 extend 调用中提取检查点" (the conv checkpoint: the
 * kernel_size - 1 rows of mixed_qkv before the boundary); [SERVE] §1.3 (alpha =
 * g_min * sigmoid(.), beta = sigmoid(.)).  Where the pages leave a step open:
 * rows of mixed_qkv are [q (H*dk) | k (H*dk) | v (H*dv)], the convolution has no
 * bias, y[t,c] = sum_j weight[c,j] * in[t - (w-1) + j, c], L2Norm is
 * x / sqrt(sum x^2 + 1e-6) over each head's dk channels after the activation.
 *   mixed_qkv    device dtype [T, C], C = H*(2*dk + dv)   in (packed sequences)
 *   conv_weight  device dtype [C, w], 2 <= w <= 8          in
 *   window_in    device dtype [n_seqs, w-1, C] or NULL     in: each sequence's
 *                window (the raw rows before it, oldest first); NULL = zeros
 *   window_out   device dtype [n_seqs, w-1, C] or NULL     out: the window after
 *                each sequence (carry it into the next call)
 *   g_logits     device dtype [T, H, dk]; beta_logits [T, H]   in
 *   g_min        g = g_min * sigmoid(g_logits) (g_min < 0)
 *   act          KDA_ACT_NONE or KDA_ACT_SILU (applied after the convolution)
 *   cu_seqlens, n_seqs, T   as kda_prefill_chunked (host)
 *   q, k, g      device dtype [T, H, dk] out; v [T, H, dv] out; beta [T, H] out
 *   ckpt_stride, conv_ckpt, num_ckpt  optional conv checkpoints: when conv_ckpt
 *                is not NULL, checkpoint c (numbered as kda_prefill_chunked
 *                numbers its states: sequence-major, then position) gets the
 *                window at its boundary, [num_ckpt, w-1, C] dtype; num_ckpt must
 *                be >= kda_num_checkpoints()
 * All tensors of one dtype (KDA_F32 or KDA_BF16); outputs must not overlap
 * inputs.  Errors: KDA_ERR_SHAPE (w, sizes, cu_seqlens), KDA_ERR_ARG (NULL
 * required pointer, act, g_min >= 0), KDA_ERR_ALIGN, KDA_ERR_ALIAS.
 */
int kda_input_prep(const void* mixed_qkv, const void* conv_weight, int w,
                   const void* window_in, void* window_out,
                   const void* g_logits, const void* beta_logits, float g_min, int act,
                   const int32_t* cu_seqlens, int n_seqs, int64_t T, int H, int dk, int dv,
                   int dtype, void* q, void* k, void* v, void* g, void* beta,
                   int ckpt_stride, void* conv_ckpt, int64_t num_ckpt, kda_stream_t stream);

/*
 * kda_pack_heads -- gather (B,H,dk,dv) states into one flat head-contiguous
 * buffer, zero-filling it past B*H*dk*dv. [SERVE] §1.5 pack_heads.
 *   S         device fp32; element (b,h,i,j) at S[b*stride_b + h*stride_h + i*dv + j]
 *   flat      device fp32 [flat_elems] out; flat_elems >= B*H*dk*dv
 * Strides are in elements and must be multiples of 4. Bit-exact copy.
 */
int kda_pack_heads(const float* S, int64_t stride_b, int64_t stride_h,
                   float* flat, int64_t flat_elems,
                   int B, int H, int dk, int dv, kda_stream_t stream);

/*
 * kda_unpack_heads -- scatter a flat head-contiguous buffer back into
 * (B,H,dk,dv) states (strided as in kda_pack_heads). [SERVE] §1.5.
 */
int kda_unpack_heads(const float* flat, float* S, int64_t stride_b, int64_t stride_h,
                     int B, int H, int dk, int dv, kda_stream_t stream);

/* ---------------------------------------------------------------------------
 * Unified page pool ([SERVE] §1.5 PagePool / PagedCache): a host-side free
 * list over a caller-owned device arena of n_pages pages of page_bytes each.
 * Pages are handed out lowest index first. Not thread-safe: one owner thread.
 * ------------------------------------------------------------------------- */
typedef struct kda_page_pool kda_page_pool;

int   kda_pool_create(void* device_base, int64_t page_bytes, int64_t n_pages,
                      kda_page_pool** pool_out);
int   kda_pool_destroy(kda_page_pool* pool);
/* take n pages of one kind; all or nothing (KDA_ERR_NOMEM leaves the pool unchanged) */
int   kda_pool_alloc(kda_page_pool* pool, int kind, int64_t n, int32_t* page_ids_out);
/* return pages; a page that is not allocated is KDA_ERR_ARG and nothing is freed */
int   kda_pool_free(kda_page_pool* pool, int64_t n, const int32_t* page_ids);
int64_t kda_pool_num_free(const kda_page_pool* pool);
int   kda_pool_page_kind(const kda_page_pool* pool, int32_t page_id);
void* kda_pool_page_ptr(const kda_page_pool* pool, int32_t page_id);
void* kda_pool_base(const kda_page_pool* pool);
int64_t kda_pool_page_bytes(const kda_page_pool* pool);

/* store_kda / load_kda ([SERVE] Tab 7): pack a (B,H,dk,dv) state into one
 * KDA page (zero-padded tail) / unpack it back. The page must be allocated
 * with kind KDA_PAGE_KDA_STATE. */
int kda_store_kda(kda_page_pool* pool, int32_t page_id, const float* S,
                  int64_t stride_b, int64_t stride_h, int B, int H, int dk, int dv,
                  kda_stream_t stream);
int kda_load_kda(const kda_page_pool* pool, int32_t page_id, float* S,
                 int64_t stride_b, int64_t stride_h, int B, int H, int dk, int dv,
                 kda_stream_t stream);

/* ---------------------------------------------------------------------------
 * Byte accounting ([SERVE] §1.1): bytes of a full state snapshot per draft
 * step over bytes of the cached projections per draft step,
 * (H dk dv) / (H (3 dk + dv + 1)). Independent of draft length and dtype.
 * Returns a negative value for non-positive sizes.
 * ------------------------------------------------------------------------- */
double kda_snapshot_cost_ratio(int H, int dk, int dv);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
