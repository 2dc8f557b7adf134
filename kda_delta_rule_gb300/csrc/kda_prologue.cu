// Input prologue of a KDA layer for prefill: causal depthwise ShortConv over the
// rows of mixed_qkv, activation, per-head L2Norm of q and k, and the gates from
// their logits ("Kimi Linear 的 KDA 缓存", section "KDA 的递推与充分状态": Q/K/V
// pass through a linear projection, a causal short convolution and an
// activation, and Q/K are L2-normalised; the serve-module demo page, §1.3:
// alpha = g_min * sigmoid(.), beta = sigmoid(.)).  The conv window carried across
// calls and the conv checkpoints at chunk-aligned boundaries are the kernel_size - 1
// raw rows before the boundary (same page, section "SGLang：从一次较长的 extend
// 调用中提取检查点").
//
// One CTA per (32-token tile of one sequence, head); each thread owns two
// adjacent channels of the head's q, k or v columns, so every row access of a
// warp is one contiguous 64- or 128-byte piece.  The tile's raw inputs and the
// w - 1 rows before it sit in registers; the convolution runs from the newest
// token down so each output overwrites an input no later output needs.  The sum
// of squares of a token's q (k) is reduced with shuffles inside the lanes of the
// group and across its warps through shared memory.  HBM-bound: every input
// element is read once (plus the w - 1 halo rows per tile) and every output
// written once.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "../../include/kda.h"

namespace kda {
namespace {

constexpr int TT = 32;     // tokens per tile
constexpr int MAXW = 8;    // largest conv kernel size (the window lives in registers)

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }

__device__ __forceinline__ int find_tile_seq(const ProSched& s, int tile) {
  int lo = 0, hi = s.n_seqs - 1;
  while (lo < hi) {                       // last n with tile_base[n] <= tile
    const int mid = (lo + hi + 1) >> 1;
    if (s.tile_base[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int DK, int DV>
struct ProCfg {
  static constexpr int NCH2 = DK + DV / 2;                  // channel pairs of one head
  static constexpr int NT = (NCH2 + 31) / 32 * 32;
  static constexpr int SEG = DK / 2 < 32 ? DK / 2 : 32;     // lanes of one reduction segment
  static constexpr int NSEG = DK / 2 / SEG;                 // segments per q (or k) group
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(ProCfg<DK, DV>::NT)
kda_prologue_kernel(const ProArgs a, const ProSched sched) {
  using Cfg = ProCfg<DK, DV>;
  __shared__ float red[2 * Cfg::NSEG][TT];
  const int tid = threadIdx.x, lane = tid & 31;
  const int h = blockIdx.y, H = a.H, w = a.w;
  const int tile = blockIdx.x;
  const int n = find_tile_seq(sched, tile);
  const int64_t s0 = sched.start[n];
  const int len = sched.len[n];
  const int pos0 = (tile - sched.tile_base[n]) * TT;       // first position of the tile in its sequence
  const int L = min(TT, len - pos0);
  const int64_t t0 = s0 + pos0;
  const int64_t C = (int64_t)H * (2 * DK + DV);

  // this thread's column pair: group 0 = q, 1 = k, 2 = v, 3 = none
  int grp, c;
  if (tid < DK / 2) { grp = 0; c = 2 * tid; }
  else if (tid < DK) { grp = 1; c = 2 * (tid - DK / 2); }
  else if (tid < Cfg::NCH2) { grp = 2; c = 2 * (tid - DK); }
  else { grp = 3; c = 0; }
  const int64_t col = grp == 0 ? (int64_t)h * DK + c
                    : grp == 1 ? (int64_t)H * DK + (int64_t)h * DK + c
                               : 2 * (int64_t)H * DK + (int64_t)h * DV + c;
  const bool mine = grp < 3;
  const T* x = reinterpret_cast<const T*>(a.mixed);
  const T* win = reinterpret_cast<const T*>(a.window_in);
  const T* wt = reinterpret_cast<const T*>(a.weight);

  // raw input of position p (< 0: the carried window, zeros without one)
  auto raw = [&](int p) -> float2 {
    if (p >= 0) return load2(x + (s0 + p) * C + col);
    if (win == nullptr) return make_float2(0.f, 0.f);
    const T* r = win + ((int64_t)n * (w - 1) + (w - 1 + p)) * C + col;
    return load2(r);
  };

  // taps by distance back from the newest input: wr[d] = weight[:, w - 1 - d]
  float2 wr[MAXW];
  float2 z[TT + MAXW - 1];                 // z[MAXW - 1 + t] = input of tile token t
  if (mine) {
#pragma unroll
    for (int d = 0; d < MAXW; ++d)
      wr[d] = d < w ? make_float2(to_f32(wt[col * w + (w - 1 - d)]), to_f32(wt[(col + 1) * w + (w - 1 - d)]))
                    : make_float2(0.f, 0.f);
#pragma unroll
    for (int t = 0; t < TT; ++t) z[MAXW - 1 + t] = t < L ? load2(x + (t0 + t) * C + col) : make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 1; r < MAXW; ++r) z[MAXW - 1 - r] = r < w ? raw(pos0 - r) : make_float2(0.f, 0.f);
    // newest token first: output t overwrites input t, which no earlier token reads
#pragma unroll
    for (int t = TT - 1; t >= 0; --t) {
      float2 y = make_float2(0.f, 0.f);
#pragma unroll
      for (int d = 0; d < MAXW; ++d) {
        y.x = fmaf(wr[d].x, z[MAXW - 1 + t - d].x, y.x);
        y.y = fmaf(wr[d].y, z[MAXW - 1 + t - d].y, y.y);
      }
      if (a.act == KDA_ACT_SILU) { y.x *= sigm(y.x); y.y *= sigm(y.y); }
      z[MAXW - 1 + t] = y;
    }
  } else {
#pragma unroll
    for (int t = 0; t < TT + MAXW - 1; ++t) z[t] = make_float2(0.f, 0.f);
  }

  // per-token sums of squares of q and k over the head
  const int gi = tid % (DK / 2), seg = gi / Cfg::SEG;
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    const float2 y = z[MAXW - 1 + t];
    float ss = grp < 2 ? fmaf(y.x, y.x, y.y * y.y) : 0.f;
#pragma unroll
    for (int off = Cfg::SEG / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (grp < 2 && (lane % Cfg::SEG) == 0) red[grp * Cfg::NSEG + seg][t] = ss;
  }
  __syncthreads();

  if (grp < 2) {
    T* out = reinterpret_cast<T*>(grp == 0 ? a.q : a.k);
    const T* gl = reinterpret_cast<const T*>(a.g_logits);
    T* gout = reinterpret_cast<T*>(a.g);
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      if (t >= L) break;
      float ss = 0.f;
#pragma unroll
      for (int sgi = 0; sgi < Cfg::NSEG; ++sgi) ss += red[grp * Cfg::NSEG + sgi][t];
      const float inv = rsqrtf(ss + a.eps);
      const float2 y = z[MAXW - 1 + t];
      const int64_t o = ((t0 + t) * H + h) * DK + c;
      store2(out + o, make_float2(y.x * inv, y.y * inv));
      if (grp == 0) {
        const float2 lg = load2(gl + o);
        store2(gout + o, make_float2(a.g_min * sigm(lg.x), a.g_min * sigm(lg.y)));
      }
    }
  } else if (grp == 2) {
    T* out = reinterpret_cast<T*>(a.v);
#pragma unroll
    for (int t = 0; t < TT; ++t)
      if (t < L) store2(out + ((t0 + t) * H + h) * DV + c, z[MAXW - 1 + t]);
  }
  if (tid < L) {
    const T* bl = reinterpret_cast<const T*>(a.beta_logits);
    T* bo = reinterpret_cast<T*>(a.beta);
    bo[(t0 + tid) * H + h] = from_f32<T>(sigm(to_f32(bl[(t0 + tid) * H + h])));
  }

  // raw windows: after the sequence (its last tile) and at every checkpoint
  // boundary b inside this tile (b - 1 in the tile); rows are positions b - w + 1 .. b - 1
  if (!mine) return;
  auto put_window = [&](T* dst, int b) {
    for (int r = 0; r < w - 1; ++r) store2(dst + (int64_t)r * C + col, raw(b - (w - 1) + r));
  };
  if (a.window_out != nullptr && pos0 + L == len)
    put_window(reinterpret_cast<T*>(a.window_out) + (int64_t)n * (w - 1) * C, len);
  if (a.conv_ckpt != nullptr && a.ckpt_stride > 0) {
    for (int b = (pos0 / a.ckpt_stride + 1) * a.ckpt_stride; b <= pos0 + L; b += a.ckpt_stride) {
      const int64_t idx = (int64_t)sched.ckpt_base[n] + b / a.ckpt_stride - 1;
      if (idx < a.num_ckpt) put_window(reinterpret_cast<T*>(a.conv_ckpt) + idx * (w - 1) * C, b);
    }
  }
}

template <int DK, int DV, typename T>
cudaError_t launch_dims(const ProArgs& a, const ProSched& sched, cudaStream_t s) {
  const int tiles = sched.tile_base[sched.n_seqs];
  if (tiles == 0) return cudaSuccess;
  kda_prologue_kernel<DK, DV, T><<<dim3((unsigned)tiles, (unsigned)a.H), ProCfg<DK, DV>::NT, 0, s>>>(a, sched);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const ProArgs& a, const ProSched& sched, cudaStream_t s) {
#define KDA_CASE(DKv, DVv) \
  if (a.dk == DKv && a.dv == DVv) return launch_dims<DKv, DVv, T>(a, sched, s);
  KDA_CASE(32, 32) KDA_CASE(32, 64) KDA_CASE(32, 128)
  KDA_CASE(64, 32) KDA_CASE(64, 64) KDA_CASE(64, 128)
  KDA_CASE(128, 32) KDA_CASE(128, 64) KDA_CASE(128, 128)
#undef KDA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prologue(const ProArgs& a, const ProSched& sched, cudaStream_t s) {
  if (a.w < 2 || a.w > MAXW) return cudaErrorInvalidValue;
  if (a.dtype == KDA_BF16) return launch_t<__nv_bfloat16>(a, sched, s);
  return launch_t<float>(a, sched, s);
}

}  // namespace kda
