// Decode step and speculative verify/replay of the KDA gated delta rule.
//
// Recurrence (one head, state S in R^{dk x dv}, rows = key channels):
//   decay first     ("Kimi Linear 的 KDA 缓存", section "KDA 的递推与充分状态"):
//       S' = Diag(e^g) S,  delta = v - S'^T k,  S = S' + beta k delta^T,  o = S^T q
//   undecayed delta (KIMI K3 Serve demo page, §1.3 kda_step):
//       delta = v - S^T k,  S = Diag(e^g) S + beta k delta^T,  o = S^T q
// Replay (KIMI K3 Serve demo page, §1.2 verify_and_replay) runs the accepted
// prefix of a draft from a clone of the committed state.
//
// Single pass over the state.  Columns of S are independent given (q,k,g,beta),
// and both orderings reduce to two row-reductions of the old state:
//   a_j = sum_i w_i S_ij   with w = e^g * k (decay first) or k (undecayed delta)
//   b_j = sum_i e^{g_i} q_i S_ij
//   delta_j = v_j - a_j,   o_j = b_j + beta (k.q) delta_j,
//   S_ij <- e^{g_i} S_ij + k_i (beta delta_j).
// So a call reads every state element once and writes it once; replay keeps
// the state in registers across all accepted steps.
//
// Thread layout per head, state stored (dk, dv): each thread owns 4 consecutive
// columns (one float4) of RPT rows; a warp-wide load covers whole rows (dv*4
// bytes contiguous), so every state access is a coalesced 128-bit access.  Row
// reductions go through warp shuffles and one shared-memory exchange per step.
// State stored transposed, (dv, dk) (the layout some kernels and state pools
// keep: "Kimi Linear 的 KDA 缓存", section "先统一记号：矩阵状态不等于完整检查点"):
// each thread owns 4 consecutive key channels of RPT rows of S^T, so loads stay
// 128-bit and coalesced; the two sums over key channels become a reduce-scatter
// across the lanes that share a row set (one warp or part of one), followed by
// one broadcast of delta through shared memory.
// Optional slot indirection (SGLang's [layers, slots, heads, d_v, d_k] buffer,
// same page, section "一个逻辑检查点如何展开"): batch row b reads the state of slot
// slot_in[b] and writes slot slot_out[b] of its layer's part of a pool (ids
// outside [0, n_slots) leave the pool untouched and the row's outputs zero).
//
// This header holds the kernel and its launch templates; kda_step_{kv,vk}_{f32,bf16}.cu
// instantiate one state layout and projection dtype each, kda_step.cu dispatches.
#pragma once
#include <atomic>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "../../include/kda.h"

namespace kda {
namespace {

template <int DK, int DV, int NW>
struct StepCfg {
  static constexpr int NT = 32 * NW;        // threads per head
  static constexpr int TPR = DV / 4;        // threads per state row
  static constexpr int RG = NT / TPR;       // row groups
  static constexpr int RPT = DK / RG;       // rows per thread
  static constexpr int STAGE = 3 * DK + DV + 4;   // floats staged per step: k, q, e^g, v, beta
  static constexpr int RED = 2 * DV + 4;          // floats per warp in the reduction buffer
  static_assert(TPR <= 32 && (32 % TPR) == 0, "dv/4 must divide 32");
  static_assert(NT % TPR == 0 && DK % RG == 0 && RPT >= 1, "bad head tiling");
};

// transposed state: rows of S^T (value channels), 4 key channels per thread
template <int DK, int DV, int NW>
struct StepCfgT {
  static constexpr int NT = 32 * NW;
  static constexpr int G = DK / 4;          // lanes per row of S^T
  static constexpr int RG = NT / G;         // row groups
  static constexpr int RPT = DV / RG;       // rows per thread
  static constexpr int NV = 2 * RPT;        // partial sums per thread per step
  static_assert(G <= 32 && (32 % G) == 0, "dk/4 must divide 32");
  static_assert(NT % G == 0 && DV % RG == 0 && RPT >= 1 && NV >= G, "bad transposed tiling");
};

// per-step k.q partials, rounded up so the reduction buffer stays 16-byte aligned
__host__ __device__ constexpr size_t kqw_floats(int steps, int nw) { return ((size_t)steps * nw + 3) / 4 * 4; }

template <int DK, int DV, int NW>
__host__ __device__ constexpr size_t step_smem_floats(int steps) {
  using C = StepCfg<DK, DV, NW>;
  return (size_t)steps * C::STAGE + kqw_floats(steps, NW) + 2 * (size_t)NW * C::RED;
}

// Decode keeps at least 16 warps resident per SM (128 registers a thread), so that
// enough state loads are in flight to cover HBM latency; replay of 32 x 32 heads
// (a warp per head, four heads per CTA) keeps at least four CTAs per SM the same way.
template <int NT_CTA, int MAXS, int HEAD_ELEMS>
constexpr int step_min_blocks() {
  return MAXS == 1 ? (NT_CTA < 512 ? 512 / NT_CTA : 1) : (HEAD_ELEMS <= 1024 && NT_CTA <= 128 ? 4 : 1);
}

// Decode with the input prologue fused into the staging: raw mixed_qkv channels of
// this head pass through the causal ShortConv (window read and shifted in place),
// the activation, per-head L2Norm of q and k, and the gates from their logits.
constexpr int kFusedMaxW = 4;   // largest conv kernel size of the fused decode (window in registers)

// Raw inputs of one head's prologue, per thread: channel slot e = 2u (q of key
// channel tid + u NT), 2u + 1 (k of it), 2 EK + u (v channel tid + u NT).
template <int DK, int DV, int NW>
struct FusedIn {
  static constexpr int NT = 32 * NW, FW = kFusedMaxW;
  static constexpr int EK = (DK + NT - 1) / NT, EV = (DV + NT - 1) / NT, NE = 2 * EK + EV;
  float xin[NE], wv[NE][FW - 1], tap[NE][FW], glg[EK], blg;
};

template <int DK, int DV, int NW>
__device__ __forceinline__ int64_t fused_col(const StepArgs& a, int hh, int tid, int e) {
  using F = FusedIn<DK, DV, NW>;
  if (e < 2 * F::EK) {
    const int i = tid + (e >> 1) * F::NT;
    return (e & 1) ? (int64_t)a.H * DK + (int64_t)hh * DK + i : (int64_t)hh * DK + i;
  }
  return 2 * (int64_t)a.H * DK + (int64_t)hh * DV + tid + (e - 2 * F::EK) * F::NT;
}
template <int DK, int DV, int NW>
__device__ __forceinline__ bool fused_has(int tid, int e) {
  using F = FusedIn<DK, DV, NW>;
  return e < 2 * F::EK ? tid + (e >> 1) * F::NT < DK : tid + (e - 2 * F::EK) * F::NT < DV;
}

// Every load of the prologue: new inputs, windows, taps and logits, issued before
// the state loads so that its arithmetic overlaps them.
template <int DK, int DV, int NW, typename T>
__device__ __forceinline__ void fused_load(const StepArgs& a, int64_t b, int hh, int64_t crow, int tid,
                                           int64_t head, FusedIn<DK, DV, NW>& f) {
  using F = FusedIn<DK, DV, NW>;
  const int w = a.conv_size;
  const int64_t Cw = (int64_t)a.H * (2 * DK + DV);
  const T* X = reinterpret_cast<const T*>(a.mixed);
  const T* Wt = reinterpret_cast<const T*>(a.conv_w);
  const T* win = reinterpret_cast<const T*>(a.conv_state) + crow * (w - 1) * Cw;
  const T* gl = reinterpret_cast<const T*>(a.g_logits);
#pragma unroll
  for (int u = 0; u < F::EK; ++u) {
    const int i = tid + u * F::NT;
    f.glg[u] = i < DK ? to_f32(gl[head * DK + i]) : 0.f;
  }
#pragma unroll
  for (int e = 0; e < F::NE; ++e) {
    const bool has = fused_has<DK, DV, NW>(tid, e);
    const int64_t col = fused_col<DK, DV, NW>(a, hh, tid, e);
    f.xin[e] = has ? to_f32(X[b * Cw + col]) : 0.f;
#pragma unroll
    for (int r = 0; r < F::FW - 1; ++r) f.wv[e][r] = has && r < w - 1 ? to_f32(win[(int64_t)r * Cw + col]) : 0.f;
#pragma unroll
    for (int j = 0; j < F::FW; ++j) f.tap[e][j] = has && j < w ? to_f32(Wt[col * w + j]) : 0.f;
  }
  f.blg = tid == 0 ? to_f32(reinterpret_cast<const T*>(a.beta_logits)[head]) : 0.f;
}

// The prologue's arithmetic: ShortConv (tap j reads the input w - 1 - j steps back),
// activation, window shift in place, per-head L2Norm of q and k, gates; then the
// step's staging (k, q, e^g, v, beta) and the k.q partials.
template <int DK, int DV, int NW, typename T>
__device__ __forceinline__ void fused_compute(const StepArgs& a, const FusedIn<DK, DV, NW>& f, int hh, int64_t crow,
                                              bool live, int tid, int lane, int warp, float* st, float* kqw,
                                              float* red, int64_t head) {
  using F = FusedIn<DK, DV, NW>;
  constexpr int EK = F::EK, EV = F::EV, NE = F::NE, FW = F::FW;
  const int w = a.conv_size;
  const int64_t Cw = (int64_t)a.H * (2 * DK + DV);
  float y[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < FW; ++j) {
      if (j < w - 1) acc = fmaf(f.tap[e][j], f.wv[e][j], acc);
      else if (j == w - 1) acc = fmaf(f.tap[e][j], f.xin[e], acc);
    }
    if (a.act == KDA_ACT_SILU) acc = __fdividef(acc, 1.f + __expf(-acc));   // about 2 ulp
    y[e] = acc;
  }
  // the window moves up one row and takes the new input
  if (live) {
    T* win = reinterpret_cast<T*>(a.conv_state) + crow * (w - 1) * Cw;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      if (!fused_has<DK, DV, NW>(tid, e)) continue;
      const int64_t col = fused_col<DK, DV, NW>(a, hh, tid, e);
#pragma unroll
      for (int r = 0; r < FW - 1; ++r)
        if (r < w - 1) win[(int64_t)r * Cw + col] = from_f32<T>(r + 1 < w - 1 ? f.wv[e][r + 1] : f.xin[e]);
    }
  }

  // per-head L2Norm of q and k
  float ssq = 0.f, ssk = 0.f;
#pragma unroll
  for (int u = 0; u < EK; ++u) {
    ssq = fmaf(y[2 * u], y[2 * u], ssq);
    ssk = fmaf(y[2 * u + 1], y[2 * u + 1], ssk);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ssq += __shfl_xor_sync(0xffffffffu, ssq, off);
    ssk += __shfl_xor_sync(0xffffffffu, ssk, off);
  }
  if (lane == 0) { red[warp] = ssq; red[NW + warp] = ssk; }
  __syncthreads();
  ssq = 0.f; ssk = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < NW; ++w2) { ssq += red[w2]; ssk += red[NW + w2]; }
  const float iq = rsqrtf(ssq + a.eps), ik = rsqrtf(ssk + a.eps);

  // stage k, q, e^g, v, beta (and keep the prepared projections if asked)
  const bool keep = live && a.q_out != nullptr;
  float kq = 0.f;
#pragma unroll
  for (int u = 0; u < EK; ++u) {
    const int i = tid + u * F::NT;
    if (i < DK) {
      const float qn = y[2 * u] * iq, kn = y[2 * u + 1] * ik;
      const float gi = __fdividef(a.g_min, 1.f + __expf(-f.glg[u]));
      st[i] = kn;
      st[DK + i] = qn;
      st[2 * DK + i] = expf(gi);
      kq = fmaf(kn, qn, kq);
      if (keep) {
        reinterpret_cast<T*>(a.q_out)[head * DK + i] = from_f32<T>(qn);
        reinterpret_cast<T*>(a.k_out)[head * DK + i] = from_f32<T>(kn);
        reinterpret_cast<T*>(a.g_out)[head * DK + i] = from_f32<T>(gi);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < EV; ++u) {
    const int j = tid + u * F::NT;
    if (j < DV) {
      st[3 * DK + j] = y[2 * EK + u];
      if (keep) reinterpret_cast<T*>(a.v_out)[head * DV + j] = from_f32<T>(y[2 * EK + u]);
    }
  }
  if (tid == 0) {
    const float bt = __fdividef(1.f, 1.f + __expf(-f.blg));
    st[3 * DK + DV] = bt;
    if (keep) reinterpret_cast<T*>(a.beta_out)[head] = from_f32<T>(bt);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
  if (lane == 0) kqw[warp] = kq;
}

template <int DK, int DV, int NW, int HPC, int MAXS, typename T, bool TRANS, bool FUSED>
__global__ void __launch_bounds__(32 * NW * HPC, (step_min_blocks<32 * NW * HPC, MAXS, DK * DV>()))
kda_step_kernel(const StepArgs a) {
  // programmatic dependent of the preceding kernel (see launch_pdl)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  using C = StepCfg<DK, DV, NW>;
  using CT = StepCfgT<DK, DV, NW>;
  constexpr int NT = C::NT;
  constexpr int TPR = TRANS ? CT::G : C::TPR, RG = TRANS ? CT::RG : C::RG, RPT = TRANS ? CT::RPT : C::RPT;
  constexpr int EK = (DK + NT - 1) / NT, EV = (DV + NT - 1) / NT;   // channels per thread

  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);

  const int tid = threadIdx.x;
  const int y = threadIdx.y;
  const int lane = tid & 31, warp = tid >> 5;
  const int c4 = tid % TPR;           // 4 consecutive elements of a stored row: 4*c4 .. 4*c4+3
  const int rg = tid / TPR;           // stored rows rg, rg+RG, ...
  const int64_t nheads = (int64_t)a.B * a.H;          // heads of one layer
  const int64_t head = (int64_t)blockIdx.x * HPC + y;  // over all stacked layers
  const bool active = head < nheads * a.layers;
  const int64_t layer = head / nheads, hl = head - layer * nheads;
  // The host picks HPC dividing H, so every head of this CTA belongs to the
  // same layer and sequence and the step count (and with it every barrier) is uniform.
  const int b = (int)((((int64_t)blockIdx.x * HPC) % nheads) / a.H);

  int n = a.steps;
  if (a.n_accepted != nullptr) {
    int na = a.n_accepted[b];
    n = na < 0 ? 0 : (na > a.steps ? a.steps : na);
  }
  // state of this head: its own, or slot slot_in[b] (read) / slot_out[b] (written)
  // of this layer's part of a [layers][n_slots][H] state pool
  int64_t srow_in = head, srow_out = head;
  bool live_state = active;
  if (a.slot_in != nullptr) {
    const int32_t si = a.slot_in[b], so = a.slot_out[b];
    live_state = active && si >= 0 && si < a.n_slots && so >= 0 && so < a.n_slots;
    const int64_t h0 = layer * a.n_slots * a.H + (hl % a.H);
    srow_in = live_state ? h0 + (int64_t)si * a.H : 0;
    srow_out = live_state ? h0 + (int64_t)so * a.H : 0;
  }
  constexpr int ROWLEN = TRANS ? DK : DV;          // floats per stored row

  // ---- fused prologue: its loads go out first, its arithmetic overlaps the state loads ----
  // conv window row: the batch row, or its slot (row 0 stands in for a skipped
  // slot; nothing is written there); head 0 stands in for a padding head
  FusedIn<DK, DV, NW> fin;
  int64_t crow = 0;
  if constexpr (FUSED) {
    crow = a.slot_in == nullptr ? (int64_t)b : live_state ? (int64_t)a.slot_in[b] : 0;
    fused_load<DK, DV, NW, T>(a, b, (int)(hl % a.H), crow, tid, active ? head : 0, fin);
  }

  // ---- issue all state loads ----
  float4 S[RPT];
  const float* Sin = a.S_in + srow_in * (int64_t)(DK * DV);
  if (live_state) {
#pragma unroll
    for (int m = 0; m < RPT; ++m) S[m] = ld_stream(Sin + (rg + RG * m) * ROWLEN + 4 * c4);
  } else {
#pragma unroll
    for (int m = 0; m < RPT; ++m) S[m] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---- stage the projections of every step this head runs ----
  const size_t per_y = step_smem_floats<DK, DV, NW>(a.steps);
  float* base = smem + y * per_y;
  float* stage = base;                                  // [steps][STAGE]
  float* kqw = stage + (size_t)a.steps * C::STAGE;      // [steps][NW]
  float* red = kqw + kqw_floats(a.steps, NW);           // [2][NW][RED]
  const T* q = reinterpret_cast<const T*>(a.q);
  const T* k = reinterpret_cast<const T*>(a.k);
  const T* v = reinterpret_cast<const T*>(a.v);
  const T* g = reinterpret_cast<const T*>(a.g);
  const T* beta = reinterpret_cast<const T*>(a.beta);
  if constexpr (FUSED) {
    static_assert(MAXS == 1, "the fused prologue is a decode path");
    fused_compute<DK, DV, NW, T>(a, fin, (int)(hl % a.H), crow, active && live_state, tid, lane, warp, stage, kqw,
                                 red, active ? head : 0);
  } else {
  // All steps' loads are issued before any is used (MAXS is 1 for decode, the
  // draft bound for replay), so staging costs one memory round trip, not one
  // per step.
  float rk[MAXS][EK], rq[MAXS][EK], rg_[MAXS][EK], rv[MAXS][EV], rb[MAXS];
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    const bool live = active && s < n;
    int slot = a.ring_start + s;                       // stored step of step s
    if (slot >= a.proj_steps) slot -= a.proj_steps;
    const int64_t hs = (layer * a.proj_steps + slot) * nheads + hl;   // (layer, step, b, h) flattened
#pragma unroll
    for (int u = 0; u < EK; ++u) {
      const int i = tid + u * NT;
      const bool ok = live && i < DK;
      rk[s][u] = ok ? to_f32(k[hs * DK + i]) : 0.f;
      rq[s][u] = ok ? to_f32(q[hs * DK + i]) : 0.f;
      rg_[s][u] = ok ? to_f32(g[hs * DK + i]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < EV; ++u) {
      const int j = tid + u * NT;
      rv[s][u] = live && j < DV ? to_f32(v[hs * DV + j]) : 0.f;
    }
    rb[s] = live && tid == 0 ? to_f32(beta[hs]) : 0.f;
  }
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    if (s < n) {
      float* st = stage + (size_t)s * C::STAGE;
      float kq = 0.f;
#pragma unroll
      for (int u = 0; u < EK; ++u) {
        const int i = tid + u * NT;
        if (i < DK) {
          st[i] = rk[s][u];
          st[DK + i] = rq[s][u];
          st[2 * DK + i] = expf(rg_[s][u]);
          kq = fmaf(rk[s][u], rq[s][u], kq);
        }
      }
#pragma unroll
      for (int u = 0; u < EV; ++u) {
        const int j = tid + u * NT;
        if (j < DV) st[3 * DK + j] = rv[s][u];
      }
      if (tid == 0) st[3 * DK + DV] = rb[s];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
      if (lane == 0) kqw[s * NW + warp] = kq;
    }
  }
  }
  __syncthreads();

  T* out = reinterpret_cast<T*>(a.out);
  const int mode = a.mode;
  for (int s = 0; s < n; ++s) {
    const float* st = stage + (size_t)s * C::STAGE;
    const float* sk = st;
    const float* sq = st + DK;
    const float* se = st + 2 * DK;
    const float bt = st[3 * DK + DV];
    if constexpr (TRANS) {
      // ---- state stored (dv, dk): this thread holds key channels 4 c4 .. 4 c4 + 3 ----
      constexpr int G = CT::G, NV = CT::NV, F = NV / G;
      float ww[4], qe[4];
      {
        const float4 k4 = *reinterpret_cast<const float4*>(sk + 4 * c4);
        const float4 e4 = *reinterpret_cast<const float4*>(se + 4 * c4);
        const float4 q4 = *reinterpret_cast<const float4*>(sq + 4 * c4);
        const bool df = mode == KDA_MODE_DECAY_FIRST;
        ww[0] = df ? e4.x * k4.x : k4.x; ww[1] = df ? e4.y * k4.y : k4.y;
        ww[2] = df ? e4.z * k4.z : k4.z; ww[3] = df ? e4.w * k4.w : k4.w;
        qe[0] = e4.x * q4.x; qe[1] = e4.y * q4.y; qe[2] = e4.z * q4.z; qe[3] = e4.w * q4.w;
      }
      // First exchange fused with the partial sums: the lower half of each row
      // set's lanes keeps the a sums (w . S) of its RPT rows, the upper half the
      // b sums (e^g q . S); each adds its partner's partial of the kept quantity.
      const bool hi = (lane & (G / 2)) != 0;
      float vals[RPT];
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const float pa = fmaf(ww[0], S[m].x, fmaf(ww[1], S[m].y, fmaf(ww[2], S[m].z, ww[3] * S[m].w)));
        const float pb = fmaf(qe[0], S[m].x, fmaf(qe[1], S[m].y, fmaf(qe[2], S[m].z, qe[3] * S[m].w)));
        vals[m] = (hi ? pb : pa) + __shfl_xor_sync(0xffffffffu, hi ? pa : pb, G / 2);
      }
      // then halve the kept sums per level (reduce-scatter) over the remaining lane bits
      int base = hi ? RPT : 0;               // index of vals[0] among [a sums, b sums]
#pragma unroll
      for (int lev = 1; (G >> (lev + 1)) >= 1; ++lev) {
        const int off = G >> (lev + 1), half = NV >> (lev + 1);
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int v2 = 0; v2 < half; ++v2) {
          const float send = up ? vals[v2] : vals[half + v2];
          const float keep = up ? vals[half + v2] : vals[v2];
          vals[v2] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        if (up) base += half;
      }
      // vals[0..F) are the full sums number base .. base + F - 1; the partner across
      // the top bit holds the other quantity of the same rows
      float other[F];
#pragma unroll
      for (int v2 = 0; v2 < F; ++v2) other[v2] = __shfl_xor_sync(0xffffffffu, vals[v2], G / 2);
      float kq = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) kq += kqw[s * NW + w];
      const float bkq = bt * kq;
      float* dl = red + rg * RPT;            // beta delta of this row set's rows
      if (base < RPT) {                      // lanes holding a (= w . S) sums
#pragma unroll
        for (int v2 = 0; v2 < F; ++v2) {
          const int m = base + v2, j = rg + RG * m;
          const float d = st[3 * DK + j] - vals[v2];
          dl[m] = bt * d;
          if (active)
            out[head * a.out_head_stride + s * a.out_step_stride + j] =
                from_f32<T>(live_state ? fmaf(bkq, d, other[v2]) : 0.f);
        }
      }
      __syncwarp();
      const float4 k4 = *reinterpret_cast<const float4*>(sk + 4 * c4);
      const float4 e4 = *reinterpret_cast<const float4*>(se + 4 * c4);
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const float bd = dl[m];
        S[m].x = fmaf(e4.x, S[m].x, k4.x * bd);
        S[m].y = fmaf(e4.y, S[m].y, k4.y * bd);
        S[m].z = fmaf(e4.z, S[m].z, k4.z * bd);
        S[m].w = fmaf(e4.w, S[m].w, k4.w * bd);
      }
      __syncwarp();                          // dl is rewritten by the next step
    } else {
      float4 pa = make_float4(0.f, 0.f, 0.f, 0.f), pb = pa;
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const int i = rg + RG * m;
        const float e = se[i];
        const float w = (mode == KDA_MODE_DECAY_FIRST) ? e * sk[i] : sk[i];
        pa = f4_fma(w, S[m], pa);
        pb = f4_fma(e * sq[i], S[m], pb);
      }
      // reduce over the lanes of this warp that share the column group
#pragma unroll
      for (int off = TPR; off < 32; off <<= 1) {
        pa.x += __shfl_xor_sync(0xffffffffu, pa.x, off); pa.y += __shfl_xor_sync(0xffffffffu, pa.y, off);
        pa.z += __shfl_xor_sync(0xffffffffu, pa.z, off); pa.w += __shfl_xor_sync(0xffffffffu, pa.w, off);
        pb.x += __shfl_xor_sync(0xffffffffu, pb.x, off); pb.y += __shfl_xor_sync(0xffffffffu, pb.y, off);
        pb.z += __shfl_xor_sync(0xffffffffu, pb.z, off); pb.w += __shfl_xor_sync(0xffffffffu, pb.w, off);
      }
      float4 A = make_float4(0.f, 0.f, 0.f, 0.f), Bq = A;
      float kq = 0.f;
      if constexpr (NW == 1) {
        // one warp per head: the butterfly above left the full sums in every lane
        A = pa;
        Bq = pb;
        kq = kqw[s];
      } else {
        float* rb = red + (size_t)(s & 1) * NW * C::RED;
        if (lane < TPR) {
          *reinterpret_cast<float4*>(rb + warp * C::RED + 4 * c4) = pa;
          *reinterpret_cast<float4*>(rb + warp * C::RED + DV + 4 * c4) = pb;
        }
        __syncthreads();
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          float4 x = *reinterpret_cast<const float4*>(rb + w * C::RED + 4 * c4);
          float4 z = *reinterpret_cast<const float4*>(rb + w * C::RED + DV + 4 * c4);
          A.x += x.x; A.y += x.y; A.z += x.z; A.w += x.w;
          Bq.x += z.x; Bq.y += z.y; Bq.z += z.z; Bq.w += z.w;
          kq += kqw[s * NW + w];
        }
      }
      const float4 vv = *reinterpret_cast<const float4*>(st + 3 * DK + 4 * c4);
      float4 d = make_float4(vv.x - A.x, vv.y - A.y, vv.z - A.z, vv.w - A.w);
      const float bkq = bt * kq;
      float4 o = make_float4(fmaf(bkq, d.x, Bq.x), fmaf(bkq, d.y, Bq.y),
                             fmaf(bkq, d.z, Bq.z), fmaf(bkq, d.w, Bq.w));
      if (!live_state) o = make_float4(0.f, 0.f, 0.f, 0.f);
      if (active && rg == 0)
        store4(out + head * a.out_head_stride + s * a.out_step_stride + 4 * c4, o);
      float4 bd = make_float4(bt * d.x, bt * d.y, bt * d.z, bt * d.w);
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const int i = rg + RG * m;
        const float e = se[i], ki = sk[i];
        S[m].x = fmaf(e, S[m].x, ki * bd.x);
        S[m].y = fmaf(e, S[m].y, ki * bd.y);
        S[m].z = fmaf(e, S[m].z, ki * bd.z);
        S[m].w = fmaf(e, S[m].w, ki * bd.w);
      }
    }
  }

  if (!active) return;
  // steps past the accepted prefix produce zero output rows
  for (int s = n; s < a.steps; ++s)
    for (int j = 4 * tid; j < DV; j += 4 * NT)
      store4(out + head * a.out_head_stride + s * a.out_step_stride + j, make_float4(0.f, 0.f, 0.f, 0.f));
  if (!live_state) return;
  float* Sout = a.S_out + srow_out * (int64_t)(DK * DV);
#pragma unroll
  for (int m = 0; m < RPT; ++m) st_stream(Sout + (rg + RG * m) * ROWLEN + 4 * c4, S[m]);
}

// ---- 32 x 32 heads: one warp per head, one state column per lane ----------------
// For the small heads of speculative replay ([SERVE] §1.2's demo shape, dk = dv = 32)
// a warp holds a whole head with lane j owning column j of S (its 32 rows in
// registers).  Both row reductions of a step are then the lane's own dot products
// (a_j = sum_i w_i S_ij, b_j = sum_i e^{g_i} q_i S_ij) with no shuffles, and the
// per-step row coefficients w_i, e^{g_i} q_i, e^{g_i}, beta k_i are shared-memory
// broadcasts staged once per call.  One warp per CTA: heads of different sequences
// run different accepted counts, and a CTA's registers come back only when its last
// warp ends, so one-warp CTAs hand each slot on as soon as its head is done; a single
// call's heads also spread over every SM (64 stacked layers 70.0 -> 68.7 us, one call
// in a CUDA graph 5.32 -> 5.19 us, against four heads per CTA).
// SPLIT = 2 gives each head two warps, 16 columns each, lane pairs (l, l + 16)
// sharing a column and taking its upper and lower 16 rows: half the dependent
// work per lane and one shuffle per sum, for calls whose heads would leave most
// warp slots of the GPU empty (a single call's latency is then the point).
constexpr int kSmallD = 32;
constexpr int kSmallHPC = 1;          // heads (warps) per CTA

template <typename T, bool TRANS, int MAXS, int SPLIT>
__global__ void __launch_bounds__(32 * kSmallHPC)
kda_step_small_kernel(const StepArgs a) {
  constexpr int D = kSmallD;
  constexpr int NCOL = D / SPLIT;                      // state columns of one warp
  constexpr int RW = D * NCOL / 32;                    // state rows of one lane
  static_assert(SPLIT == 1 || SPLIT == 2, "one or two warps per head");
  __shared__ float4 coef[kSmallHPC][MAXS][4][D / 4];   // per step: w, e^g q, e^g, beta k (rows 0..31)
  // launched as a programmatic dependent of the preceding kernel: the next launch
  // may be placed at once, and nothing is read before the preceding kernel's
  // writes are complete and visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t nheads = (int64_t)a.B * a.H;
  const int64_t unit = (int64_t)blockIdx.x * kSmallHPC + w;   // (head, column part)
  const int64_t head = unit / SPLIT;                          // over all stacked layers
  if (head >= nheads * a.layers) return;                      // whole warps leave; no CTA barrier follows
  const int j = (int)(unit % SPLIT) * NCOL + lane % NCOL;     // this lane's state column
  const int r0 = (lane / NCOL) * RW;                          // and its first row
  const int64_t layer = head / nheads, hl = head - layer * nheads;
  const int b = (int)(hl / a.H);
  int n = a.steps;
  if (a.n_accepted != nullptr) {
    const int na = a.n_accepted[b];
    n = na < 0 ? 0 : (na > a.steps ? a.steps : na);
  }
  int64_t srow_in = head, srow_out = head;
  bool live_state = true;
  if (a.slot_in != nullptr) {
    const int32_t si = a.slot_in[b], so = a.slot_out[b];
    live_state = si >= 0 && si < a.n_slots && so >= 0 && so < a.n_slots;
    const int64_t h0 = layer * a.n_slots * a.H + (hl % a.H);
    srow_in = live_state ? h0 + (int64_t)si * a.H : 0;
    srow_out = live_state ? h0 + (int64_t)so * a.H : 0;
  }
  // ---- state: rows r0 .. r0 + RW - 1 of column j (stored (dk, dv): coalesced
  // row segments; stored (dv, dk): a contiguous piece of row j of S^T) ----
  float S[RW];
  const float* Sin = a.S_in + srow_in * (int64_t)(D * D);
  if (live_state) {
    if constexpr (TRANS) {
#pragma unroll
      for (int i = 0; i < RW; i += 4) {
        const float4 x = *reinterpret_cast<const float4*>(Sin + j * D + r0 + i);
        S[i] = x.x; S[i + 1] = x.y; S[i + 2] = x.z; S[i + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < RW; ++i) S[i] = Sin[(r0 + i) * D + j];
    }
  } else {
#pragma unroll
    for (int i = 0; i < RW; ++i) S[i] = 0.f;
  }
  // ---- projections of every step: lane i brings key channel i, and value channel j ----
  const T* q = reinterpret_cast<const T*>(a.q);
  const T* k = reinterpret_cast<const T*>(a.k);
  const T* v = reinterpret_cast<const T*>(a.v);
  const T* g = reinterpret_cast<const T*>(a.g);
  const T* beta = reinterpret_cast<const T*>(a.beta);
  float rk[MAXS], rq[MAXS], rg[MAXS], rv[MAXS], rb[MAXS];
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    const bool live = s < n;
    int slot = a.ring_start + s;                       // stored step of step s
    if (slot >= a.proj_steps) slot -= a.proj_steps;
    const int64_t hs = (layer * a.proj_steps + slot) * nheads + hl;   // (layer, step, b, h) flattened
    rk[s] = live ? to_f32(k[hs * D + lane]) : 0.f;
    rq[s] = live ? to_f32(q[hs * D + lane]) : 0.f;
    rg[s] = live ? to_f32(g[hs * D + lane]) : 0.f;
    rv[s] = live ? to_f32(v[hs * D + j]) : 0.f;
    rb[s] = live ? to_f32(beta[hs]) : 0.f;
  }
  // per-step row coefficients of the accepted steps
  float kq[MAXS];
  const bool df = a.mode == KDA_MODE_DECAY_FIRST;
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    if (s < n) {
      const float e = expf(rg[s]);
      float* c = reinterpret_cast<float*>(coef[w][s]);
      c[lane] = df ? e * rk[s] : rk[s];
      c[D + lane] = e * rq[s];
      c[2 * D + lane] = e;
      c[3 * D + lane] = rb[s] * rk[s];
    }
    kq[s] = rk[s] * rq[s];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {          // the steps' k.q butterflies, interleaved
#pragma unroll
    for (int s = 0; s < MAXS; ++s) kq[s] += __shfl_xor_sync(0xffffffffu, kq[s], off);
  }
  __syncwarp();
  // ---- the accepted steps ----
  T* out = reinterpret_cast<T*>(a.out);
  T* orow = out + head * a.out_head_stride + j;
  const bool writer = r0 == 0;                         // one lane per column writes the outputs
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    if (s < n) {
      const float4* cw = coef[w][s][0];
      const float4* cq = coef[w][s][1];
      const float4* ce = coef[w][s][2];
      const float4* ck = coef[w][s][3];
      // four independent chains per sum over the lane's rows, two per packed fp32
      // (two-lane) fused multiply-add: the roundings of scalar ones in half the
      // instructions; at SPLIT = 2 the partner lane's sum over the other 16 rows of
      // the column is added last (so the two forms differ in the last bits)
      float2 a01 = make_float2(0.f, 0.f), a23 = a01, b01 = a01, b23 = a01;
#pragma unroll
      for (int i4 = 0; i4 < RW / 4; ++i4) {
        const float4 x = cw[r0 / 4 + i4], y = cq[r0 / 4 + i4];
        const int i = 4 * i4;
        const float2 s01 = make_float2(S[i], S[i + 1]), s23 = make_float2(S[i + 2], S[i + 3]);
        a01 = __ffma2_rn(make_float2(x.x, x.y), s01, a01);
        a23 = __ffma2_rn(make_float2(x.z, x.w), s23, a23);
        b01 = __ffma2_rn(make_float2(y.x, y.y), s01, b01);
        b23 = __ffma2_rn(make_float2(y.z, y.w), s23, b23);
      }
      float sa = (a01.x + a01.y) + (a23.x + a23.y), sb = (b01.x + b01.y) + (b23.x + b23.y);
      if constexpr (SPLIT == 2) {         // lanes l and l ^ 16 add the same two terms
        sa += __shfl_xor_sync(0xffffffffu, sa, 16);
        sb += __shfl_xor_sync(0xffffffffu, sb, 16);
      }
      const float d = rv[s] - sa;
      const float o = fmaf(rb[s] * kq[s], d, sb);
      if (writer) orow[s * a.out_step_stride] = from_f32<T>(live_state ? o : 0.f);
      const float2 d2 = make_float2(d, d);
#pragma unroll
      for (int i4 = 0; i4 < RW / 4; ++i4) {
        const float4 e4 = ce[r0 / 4 + i4], k4 = ck[r0 / 4 + i4];
        const int i = 4 * i4;
        const float2 lo = __ffma2_rn(make_float2(e4.x, e4.y), make_float2(S[i], S[i + 1]),
                                     __fmul2_rn(make_float2(k4.x, k4.y), d2));
        const float2 hi = __ffma2_rn(make_float2(e4.z, e4.w), make_float2(S[i + 2], S[i + 3]),
                                     __fmul2_rn(make_float2(k4.z, k4.w), d2));
        S[i] = lo.x;
        S[i + 1] = lo.y;
        S[i + 2] = hi.x;
        S[i + 3] = hi.y;
      }
    }
  }
  // steps past the accepted prefix produce zero output rows
  if (writer)
    for (int s = n; s < a.steps; ++s) orow[s * a.out_step_stride] = from_f32<T>(0.f);
  if (!live_state) return;
  float* Sout = a.S_out + srow_out * (int64_t)(D * D);
  if constexpr (TRANS) {
#pragma unroll
    for (int i = 0; i < RW; i += 4)
      *reinterpret_cast<float4*>(Sout + j * D + r0 + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < RW; ++i) Sout[(r0 + i) * D + j] = S[i];
  }
}

// Launch a step kernel as a programmatic dependent of the preceding kernel on an
// eager stream: back-to-back calls overlap one kernel's launch with the previous
// one's run (each kernel waits on the grid dependency before its first read).
// Inside a stream capture the plain launch is kept: replayed graphs pipeline
// their kernel nodes better without it.
template <typename Kern>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const StepArgs& a) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    cap = cudaStreamCaptureStatusActive;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cap == cudaStreamCaptureStatusNone ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// SM count of the current device, looked up once per device.
inline cudaError_t step_device_sms(int* sms) {
  static std::atomic<int> cache[64];            // 0 = not looked up yet
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < 64;
  if (cached && (*sms = cache[dev].load(std::memory_order_relaxed)) > 0) return cudaSuccess;
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && cached) cache[dev].store(*sms, std::memory_order_relaxed);
  return e;
}

template <typename T, bool TRANS, int SPLIT>
cudaError_t launch_small_split(const StepArgs& a, cudaStream_t s) {
  const int64_t units = (int64_t)a.B * a.H * a.layers * SPLIT;
  const dim3 grid((unsigned)((units + kSmallHPC - 1) / kSmallHPC)), block(32 * kSmallHPC);
  if (a.steps <= 1) return launch_pdl(kda_step_small_kernel<T, TRANS, 1, SPLIT>, grid, block, 0, s, a);
  if (a.steps <= 8) return launch_pdl(kda_step_small_kernel<T, TRANS, 8, SPLIT>, grid, block, 0, s, a);
  return launch_pdl(kda_step_small_kernel<T, TRANS, KDA_MAX_DRAFT, SPLIT>, grid, block, 0, s, a);
}

template <typename T, bool TRANS>
cudaError_t launch_small(const StepArgs& a, cudaStream_t s) {
  // two warps per head while the doubled grid stays within 16 warps per SM
  int sms = 0;
  cudaError_t e = step_device_sms(&sms);
  if (e != cudaSuccess) return e;
  const int64_t heads = (int64_t)a.B * a.H * a.layers;
  return 2 * heads <= 16 * (int64_t)sms ? launch_small_split<T, TRANS, 2>(a, s) : launch_small_split<T, TRANS, 1>(a, s);
}

template <int DK, int DV, typename T, bool TRANS, bool FUSED>
cudaError_t launch_dims(const StepArgs& a, cudaStream_t s) {
  if constexpr (DK == kSmallD && DV == kSmallD && !FUSED) return launch_small<T, TRANS>(a, s);
  // rows per thread 16 where the head is big enough; at least 128 threads per CTA
  constexpr int TPR = DV / 4;
  constexpr int NW0 = (DK * TPR) / (16 * 32);
  constexpr int NW = NW0 < 1 ? 1 : NW0;
  constexpr int NT = 32 * NW;
  constexpr int HMAX = NT >= 128 ? 1 : 128 / NT;   // heads per CTA: at least 128 threads
  const int64_t nheads = (int64_t)a.B * a.H;
  int hpc = 1;
  while (hpc < HMAX && (a.H % (hpc * 2)) == 0) hpc *= 2;
  size_t smem = step_smem_floats<DK, DV, NW>(a.steps) * sizeof(float);
  auto run = [&](auto kern, int HPCv) -> cudaError_t {
    size_t total = smem * HPCv;
    if (total > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)total);
      if (e != cudaSuccess) return e;
    }
    dim3 block(NT, HPCv);
    int64_t grid = (nheads * a.layers + HPCv - 1) / HPCv;
    return launch_pdl(kern, dim3((unsigned)grid), block, total, s, a);
  };
  if (FUSED || a.steps == 1) {
    if constexpr (HMAX >= 4) {
      if (hpc >= 4) return run(kda_step_kernel<DK, DV, NW, 4, 1, T, TRANS, FUSED>, 4);
    }
    if constexpr (HMAX >= 2) {
      if (hpc >= 2) return run(kda_step_kernel<DK, DV, NW, 2, 1, T, TRANS, FUSED>, 2);
    }
    return run(kda_step_kernel<DK, DV, NW, 1, 1, T, TRANS, FUSED>, 1);
  }
  // drafts of up to 8 steps (the common case) keep half the staging registers
  if (a.steps <= 8) {
    if constexpr (HMAX >= 4) {
      if (hpc >= 4) return run(kda_step_kernel<DK, DV, NW, 4, 8, T, TRANS, false>, 4);
    }
    if constexpr (HMAX >= 2) {
      if (hpc >= 2) return run(kda_step_kernel<DK, DV, NW, 2, 8, T, TRANS, false>, 2);
    }
    return run(kda_step_kernel<DK, DV, NW, 1, 8, T, TRANS, false>, 1);
  }
  if constexpr (HMAX >= 4) {
    if (hpc >= 4) return run(kda_step_kernel<DK, DV, NW, 4, KDA_MAX_DRAFT, T, TRANS, false>, 4);
  }
  if constexpr (HMAX >= 2) {
    if (hpc >= 2) return run(kda_step_kernel<DK, DV, NW, 2, KDA_MAX_DRAFT, T, TRANS, false>, 2);
  }
  return run(kda_step_kernel<DK, DV, NW, 1, KDA_MAX_DRAFT, T, TRANS, false>, 1);
}

template <typename T, bool TRANS>
cudaError_t launch_layout(const StepArgs& a, cudaStream_t s) {
#define KDA_CASE(DKv, DVv) \
  if (a.dk == DKv && a.dv == DVv)                                     \
    return a.mixed != nullptr ? launch_dims<DKv, DVv, T, TRANS, true>(a, s) \
                              : launch_dims<DKv, DVv, T, TRANS, false>(a, s);
  KDA_CASE(32, 32) KDA_CASE(32, 64) KDA_CASE(32, 128)
  KDA_CASE(64, 32) KDA_CASE(64, 64) KDA_CASE(64, 128)
  KDA_CASE(128, 32) KDA_CASE(128, 64) KDA_CASE(128, 128)
#undef KDA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace kda
