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
// This header holds the kernel and its launch templates; kda_prologue_{f32,bf16}.cu
// instantiate one dtype each (with the dtype's copy of the device error word),
// kda_prologue.cu dispatches.
//
// One CTA per (16-token tile of one sequence, head), the CTAs of one tile
// adjacent in the grid.  One thread issues four TMA copies: the head's q, k and v
// columns of mixed_qkv for the tile plus the w - 1 rows before it, and the tile's
// gate logits, all into shared memory, completion on one mbarrier (bounded wait).
// The first tile of a sequence then overwrites its halo rows with the carried
// window.  Each lane owns eight adjacent channels (one 16-byte shared-memory read
// and one 16-byte global store per token) of q, k, v or the gate logits and walks
// the tile's tokens in order with the conv window rolling through registers:
// convolution, activation, for q and k the L2Norm (its sum of squares reduced
// over the row's lanes with shuffles), store.  Window and conv-checkpoint rows
// are copied raw from shared memory.  HBM-bound: every input element is read once
// (plus the halo rows, mostly from L2) and every output written once.
#pragma once
#include <climits>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc.cuh"
#include "kda_tmap.h"
#include "../../include/kda.h"

namespace kda {
namespace {

using tc::mbar_init;
using tc::mbar_init_fence;
using tc::mbar_expect_tx;
using tc::mbar_wait;
using tc::smem_u32;
using tc::tma_load_2d;

constexpr int TT = kPrologueTile;  // tokens per tile
constexpr int VEC = 8;             // channels per lane
constexpr int MAXW = 8;            // largest conv kernel size

// sigmoid through the hardware exp2 and reciprocal (about 2 ulp; 0 for very
// negative x, where 1 + e^-x overflows)
__device__ __forceinline__ float sigm(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

// hardware tanh (relative error about 2^-11, below the 2^-9 of a bf16 store)
__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// sigmoid and SiLU for outputs stored as T: sigmoid(x) = (1 + tanh(x / 2)) / 2 when
// the result is rounded to bf16, the exp2/reciprocal form for fp32 outputs
template <typename T> __device__ __forceinline__ float sigm_out(float x) {
  if constexpr (sizeof(T) == 2) return fmaf(0.5f, tanh_hw(0.5f * x), 0.5f);
  else return sigm(x);
}
template <typename T> __device__ __forceinline__ float silu_out(float x) {
  if constexpr (sizeof(T) == 2) { const float hx = 0.5f * x; return fmaf(hx, tanh_hw(hx), hx); }
  else return __fdividef(x, 1.f + __expf(-x));
}

__device__ __forceinline__ int find_tile_seq(const ProSched& s, int tile) {
  int lo = 0, hi = s.n_seqs - 1;
  while (lo < hi) {                       // last n with tile_base[n] <= tile
    const int mid = (lo + hi + 1) >> 1;
    if (s.tile_base[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct ProMaps {
  CUtensorMap qk;   // mixed [T][C], box DK x (TT + W - 1)
  CUtensorMap v;    // mixed [T][C], box DV x (TT + W - 1)
  CUtensorMap g;    // g_logits [T][H * DK], box DK x TT
};

__host__ __device__ constexpr int up128(int x) { return (x + 127) / 128 * 128; }

// lanes of one head: q [0, NQ), k [NQ, 2 NQ), v [2 NQ, 2 NQ + NV), gate logits after
template <int DK, int DV, int W, typename T>
struct ProCfg {
  static constexpr int NQ = DK / VEC, NV = DV / VEC;
  static constexpr int LH = 3 * NQ + NV;
  static constexpr int NT = (LH + 31) / 32 * 32;
  static constexpr int HALO = W - 1, ROWS = TT + HALO;
  static constexpr int ES = (int)sizeof(T);
  static constexpr int QB = ROWS * DK * ES, VB = ROWS * DV * ES, GB = TT * DK * ES;
  static constexpr int OQ = 0, OK = up128(QB), OV = OK + up128(QB), OG = OV + up128(VB);
  static constexpr int SMEM = OG + up128(GB) + 128;           // + alignment slack
  static constexpr uint32_t TX = 2 * QB + VB + GB;            // bytes the four copies deliver
  static_assert(2 * NQ <= 32, "q and k rows of a head share one warp");
};

// W: the conv kernel size, or MAXW for any size up to MAXW (taps past w are zero);
// SILU: the activation after the convolution
template <int DK, int DV, int W, bool SILU, typename T>
__global__ void __launch_bounds__(ProCfg<DK, DV, W, T>::NT)
kda_prologue_kernel(const ProArgs a, const ProSched sched, const __grid_constant__ ProMaps maps) {
  using Cfg = ProCfg<DK, DV, W, T>;
  constexpr int NQ = Cfg::NQ, NV = Cfg::NV, HALO = Cfg::HALO;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  __shared__ uint64_t bar_word;
  const uint32_t bar = smem_u32(&bar_word);

  const int l = threadIdx.x;
  const int H = a.H, w = W == MAXW ? a.w : W;
  const int h = (int)(blockIdx.x % (unsigned)H), tile = (int)(blockIdx.x / (unsigned)H);
  const int n = find_tile_seq(sched, tile);
  const int64_t s0 = sched.start[n];
  const int len = sched.len[n];
  const int pos0 = (tile - sched.tile_base[n]) * TT;       // first position of the tile in its sequence
  const int L = min(TT, len - pos0);
  const int64_t t0 = s0 + pos0;
  const int64_t C = (int64_t)H * (2 * DK + DV);

  if (l == 0) {
    mbar_init(bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (l == 0) {
    mbar_expect_tx(bar, Cfg::TX);
    const int y0 = (int)(t0 - HALO);                       // may be negative: rows there read as zero
    tma_load_2d(smem_u32(sm + Cfg::OQ), &maps.qk, h * DK, y0, bar);
    tma_load_2d(smem_u32(sm + Cfg::OK), &maps.qk, H * DK + h * DK, y0, bar);
    tma_load_2d(smem_u32(sm + Cfg::OV), &maps.v, 2 * H * DK + h * DV, y0, bar);
    tma_load_2d(smem_u32(sm + Cfg::OG), &maps.g, h * DK, (int)t0, bar);
  }

  // role: 0 q, 1 k, 2 v (conv lanes), 3 gate logits, 4 none
  int role, c;
  if (l < NQ) { role = 0; c = VEC * l; }
  else if (l < 2 * NQ) { role = 1; c = VEC * (l - NQ); }
  else if (l < 2 * NQ + NV) { role = 2; c = VEC * (l - 2 * NQ); }
  else if (l < 3 * NQ + NV) { role = 3; c = VEC * (l - 2 * NQ - NV); }
  else { role = 4; c = 0; }
  const bool conv_lane = role < 3;
  const int64_t col = role == 0 ? (int64_t)h * DK + c
                    : role == 1 ? (int64_t)H * DK + (int64_t)h * DK + c
                                : 2 * (int64_t)H * DK + (int64_t)h * DV + c;
  const int width = role == 2 ? DV : DK;                   // elements per shared-memory row of this lane's tile
  const T* tile_s = reinterpret_cast<const T*>(sm + (role == 0 ? Cfg::OQ : role == 1 ? Cfg::OK
                                                     : role == 2 ? Cfg::OV : Cfg::OG)) + c;
  T* dst = nullptr;
  int64_t dstride = 0;
  if (conv_lane) {
    const int64_t dcol = role == 2 ? (int64_t)h * DV + c : (int64_t)h * DK + c;
    dstride = role == 2 ? (int64_t)H * DV : (int64_t)H * DK;
    dst = reinterpret_cast<T*>(role == 0 ? a.q : role == 1 ? a.k : a.v) + t0 * dstride + dcol;
  } else if (role == 3) {
    dstride = (int64_t)H * DK;
    dst = reinterpret_cast<T*>(a.g) + (t0 * H + h) * DK + c;
  }

  // while the copies run: taps by distance back (tap[0] multiplies the newest input), beta.
  // For bf16 outputs with SiLU the taps are halved (exact): the convolution then
  // yields x / 2, the argument SiLU(x) = x/2 + x/2 tanh(x/2) starts from.
  constexpr bool HALF_TAPS = SILU && sizeof(T) == 2;
  float tap[W][VEC];
  if (conv_lane) {
    const T* wt = reinterpret_cast<const T*>(a.weight);
    if constexpr (W != MAXW) {
      // the eight channels' taps are VEC * W contiguous elements (16-byte multiple, aligned)
      float wv[VEC * W];
#pragma unroll
      for (int i = 0; i < W; ++i) {
        float v8[VEC];
        load8(wt + col * W + VEC * i, v8);
#pragma unroll
        for (int e = 0; e < VEC; ++e) wv[VEC * i + e] = v8[e];
      }
#pragma unroll
      for (int d = 0; d < W; ++d)
#pragma unroll
        for (int e = 0; e < VEC; ++e) tap[d][e] = (HALF_TAPS ? 0.5f : 1.f) * wv[e * W + (W - 1 - d)];
    } else {
#pragma unroll
      for (int d = 0; d < W; ++d)
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          tap[d][e] = d < w ? (HALF_TAPS ? 0.5f : 1.f) * to_f32(wt[(col + e) * w + (w - 1 - d)]) : 0.f;
    }
  }
  for (int t = l; t < L; t += Cfg::NT) {
    const T* bl = reinterpret_cast<const T*>(a.beta_logits);
    reinterpret_cast<T*>(a.beta)[(t0 + t) * H + h] = from_f32<T>(sigm_out<T>(to_f32(bl[(t0 + t) * H + h])));
  }

  if (!mbar_wait(bar, 0)) {
    mbar_wait(bar, 0);     // the copies may still be landing: wait once more before leaving
    return;
  }
  // a sequence's first tile: the halo rows before it are the carried window (or zeros)
  if (pos0 == 0 && conv_lane) {
    const T* win = reinterpret_cast<const T*>(a.window_in);
#pragma unroll
    for (int d = 1; d < W; ++d) {
      if (d >= w) continue;
      float v8[VEC];
      if (win != nullptr) load8(win + ((int64_t)n * (w - 1) + (w - 1 - d)) * C + col, v8);
      else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v8[e] = 0.f;
      }
      store8(const_cast<T*>(tile_s) + (HALO - d) * width, v8);
    }
  }

  // conv window as a ring of W - 1 rows: the input d tokens before token t sits in
  // slot (t - d) mod (W - 1); tokens run in groups of W - 1 so every slot index is static
  constexpr int R = W - 1;
  float ring[R][VEC];
  if (conv_lane) {
#pragma unroll
    for (int d = 1; d < W; ++d) load8(tile_s + (HALO - d) * width, ring[(R - d % R) % R]);
  }
  const int row0 = role == 3 ? 0 : HALO;                   // shared-memory row of tile token 0
  int next_ck = (a.conv_ckpt != nullptr && a.ckpt_stride > 0) ? (pos0 / a.ckpt_stride + 1) * a.ckpt_stride : INT_MAX;
  // A sequence end is always a tile's last token, and so is every checkpoint
  // boundary when the stride is a multiple of the tile; only other strides need
  // the boundary test at every token.
  const bool ck_inside = a.conv_ckpt != nullptr && a.ckpt_stride > 0 && (a.ckpt_stride % TT) != 0;
  T* dptr = dst;
  for (int tb = 0; tb < L; tb += R) {
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int t = tb + u;
      if (t >= L) break;                                   // uniform across the CTA
      float y[VEC], xs[VEC];
      if (role < 4) load8(tile_s + (row0 + t) * width, xs);
      if (conv_lane) {
        // channel pairs through packed fp32 multiplies and fused multiply-adds
        // (the roundings of the scalar ones)
        float2 acc2[VEC / 2];
#pragma unroll
        for (int e = 0; e < VEC; e += 2)
          acc2[e / 2] = __fmul2_rn(make_float2(tap[0][e], tap[0][e + 1]), make_float2(xs[e], xs[e + 1]));
#pragma unroll
        for (int d = 1; d < W; ++d) {
          const int sl = ((u - d) % R + R) % R;
#pragma unroll
          for (int e = 0; e < VEC; e += 2)
            acc2[e / 2] = __ffma2_rn(make_float2(tap[d][e], tap[d][e + 1]),
                                     make_float2(ring[sl][e], ring[sl][e + 1]), acc2[e / 2]);
        }
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
          const float2 acc = acc2[e / 2];
          if constexpr (HALF_TAPS) {                           // acc = x / 2
            const float2 th = make_float2(tanh_hw(acc.x), tanh_hw(acc.y));
            const float2 r2 = __ffma2_rn(acc, th, acc);
            y[e] = r2.x;
            y[e + 1] = r2.y;
          } else {
            y[e] = SILU ? silu_out<T>(acc.x) : acc.x;
            y[e + 1] = SILU ? silu_out<T>(acc.y) : acc.y;
          }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) ring[u][e] = xs[e];   // the oldest row leaves, token t enters
      } else {
        if constexpr (sizeof(T) == 2) {
          // g_min sigmoid(x) = g_min/2 + g_min/2 tanh(x/2) in one rounding
          const float hg = 0.5f * a.g_min;
          const float2 hg2 = make_float2(hg, hg), h2 = make_float2(0.5f, 0.5f);
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            const float2 x2 = __fmul2_rn(h2, make_float2(xs[e], xs[e + 1]));
            const float2 r2 = __ffma2_rn(hg2, make_float2(tanh_hw(x2.x), tanh_hw(x2.y)), hg2);
            y[e] = r2.x;
            y[e + 1] = r2.y;
          }
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e) y[e] = a.g_min * sigm_out<T>(xs[e]);
        }
      }
      // L2Norm of q and k: the row's lanes are NQ consecutive lanes of warp 0 (the
      // other warps hold only v and gate lanes and skip it)
      if (l < 32) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
        for (int off = NQ / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (role < 2) {
          const float inv = rsqrtf(ss + a.eps);
          const float2 inv2 = make_float2(inv, inv);
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            const float2 r2 = __fmul2_rn(make_float2(y[e], y[e + 1]), inv2);
            y[e] = r2.x;
            y[e + 1] = r2.y;
          }
        }
      }
      if (role < 4) store8(dptr, y);
      dptr += dstride;

      // raw windows after position b = pos0 + t + 1 (the end of the sequence, every
      // conv checkpoint boundary): rows b - w + 1 .. b - 1, oldest first
      const int b = pos0 + t + 1;
      if (!ck_inside && t != L - 1) continue;
      const bool at_end = a.window_out != nullptr && b == len;
      const bool at_ck = b == next_ck;
      if (at_ck) next_ck += a.ckpt_stride;
      if (conv_lane && (at_end || at_ck)) {
        const int64_t idx = at_ck ? (int64_t)sched.ckpt_base[n] + b / a.ckpt_stride - 1 : 0;
        for (int r = 0; r < w - 1; ++r) {
          const T* srow = tile_s + (HALO + t + 1 - (w - 1) + r) * width;
#pragma unroll
          for (int half = 0; half < (int)sizeof(T) / 2; ++half) {   // 16 bytes each: 8 bf16 or 4 fp32
            const int off = half * (VEC * 2 / (int)sizeof(T));
            const uint4 raw = *reinterpret_cast<const uint4*>(srow + off);
            if (at_end)
              *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.window_out) + ((int64_t)n * (w - 1) + r) * C + col + off) =
                  raw;
            if (at_ck && idx < a.num_ckpt)
              *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.conv_ckpt) + (idx * (w - 1) + r) * C + col + off) = raw;
          }
        }
      }
    }
  }
}

template <int DK, int DV, int W, typename T>
cudaError_t launch_w(const ProArgs& a, const ProSched& sched, const ProMaps& maps, unsigned grid, cudaStream_t s) {
  using Cfg = ProCfg<DK, DV, W, T>;
  auto kern = a.act == KDA_ACT_SILU ? kda_prologue_kernel<DK, DV, W, true, T> : kda_prologue_kernel<DK, DV, W, false, T>;
  if (Cfg::SMEM > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, Cfg::NT, Cfg::SMEM, s>>>(a, sched, maps);
  return cudaGetLastError();
}

template <int DK, int DV, typename T>
cudaError_t launch_dims(const ProArgs& a, const ProSched& sched, int64_t T_rows, cudaStream_t s) {
  const int tiles = sched.tile_base[sched.n_seqs];
  if (tiles == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((int64_t)a.H * tiles);
  const int W = a.w <= 4 ? a.w : MAXW;
  const int64_t C = (int64_t)a.H * (2 * DK + DV);
  ProMaps maps;
  const int es = (int)sizeof(T);
  if (!make_map_2d(&maps.qk, a.mixed, T_rows, C, es, DK, TT + W - 1, false) ||
      !make_map_2d(&maps.v, a.mixed, T_rows, C, es, DV, TT + W - 1, false) ||
      !make_map_2d(&maps.g, a.g_logits, T_rows, (int64_t)a.H * DK, es, DK, TT, false))
    return cudaErrorInvalidValue;
  switch (W) {
    case 2: return launch_w<DK, DV, 2, T>(a, sched, maps, grid, s);
    case 3: return launch_w<DK, DV, 3, T>(a, sched, maps, grid, s);
    case 4: return launch_w<DK, DV, 4, T>(a, sched, maps, grid, s);
    default: return launch_w<DK, DV, MAXW, T>(a, sched, maps, grid, s);
  }
}

template <typename T>
cudaError_t launch_t(const ProArgs& a, const ProSched& sched, cudaStream_t s) {
#define KDA_CASE(DKv, DVv) \
  if (a.dk == DKv && a.dv == DVv) return launch_dims<DKv, DVv, T>(a, sched, a.T, s);
  KDA_CASE(32, 32) KDA_CASE(32, 64) KDA_CASE(32, 128)
  KDA_CASE(64, 32) KDA_CASE(64, 64) KDA_CASE(64, 128)
  KDA_CASE(128, 32) KDA_CASE(128, 64) KDA_CASE(128, 128)
#undef KDA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace kda
