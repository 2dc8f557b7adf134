// Chunked prefill of the KDA gated delta rule on tcgen05 tensor cores (bf16
// operands, fp32 accumulation and state), dk = 128, dv in {64, 128}.
//
// Math ("Kimi Linear 的 KDA 缓存", section "预填充为什么能分块并行": every
// token's transition is a diagonal minus a rank-one matrix; a 64-token chunk
// compresses into WY/UT form with a small lower-triangular solve).  Per chunk
// and head, with Gamma_r the inclusive per-channel cumsum of g inside the chunk
// and G_r = Gamma_r (decay first) or Gamma_{r-1} (undecayed delta):
//   A[r,s] = beta_s <k_r, k_s e^{G_r - Gamma_s}>   (s < r),  T = (I + A)^{-1}
//   P[r,s] = <q_r, k_s e^{Gamma_r - Gamma_s}>       (s <= r)
//   W = T (k e^{G}),  U = T V                        (WY representation)
//   Delta' = beta (U - W S)                          (needs the state)
//   O = (q e^{Gamma}) S + P Delta'
//   S <- e^{Gamma_C} S + (k e^{Gamma_C - Gamma})^T Delta'
// Two kernels:
//  * chunk prep, one CTA per (chunk, head), all chunks in parallel: gates,
//    A and P on tcgen05, the UT solve in shared memory, W and U on tcgen05.
//    It writes, per chunk and head, a pre-swizzled image of every operand the
//    state recurrence needs (the "chunk image") into the caller's workspace.
//  * chain, one CTA per (sequence, head, 32- or 64-column slice of dv), walking the
//    chunks in order: bulk-async (TMA) copies of the chunk images into a
//    two-stage ring, three tcgen05 contractions per chunk with the fp32 state
//    in registers, outputs and chunk-aligned checkpoints straight to memory
//    ("SGLang：从一次较长的 extend 调用中提取检查点"; pages in pack_heads layout,
//    KIMI K3 Serve demo page §1.5).
// Pairwise decays are split at a reference token per 16-token column block
// (its 8th token), so every exponential factor stays below e^{8 |g_min|}:
// finite in bf16/fp32 for g >= -10.
#include <cuda.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc.cuh"
#include "kda_tmap.h"
#include "../../include/kda.h"

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <mutex>
#include <type_traits>

namespace kda {
namespace {
using namespace tc;

constexpr int C = 64;
constexpr int DKT = 128;

// ---- chunk image: byte offsets inside the image of one (chunk, head) -------
// WQ: K-major [128 rows][128]: rows 0-63 = -beta W, rows 64-127 = q e^{Gamma}
// KB: MN-major (mn = dk, K = 64 tokens): k e^{Gamma_C - Gamma}
// P : K-major [64 rows][64]: P (masked)
// U : [dv/64][64 rows][64] bf16: beta U, 16-byte chunk c of row r at c ^ (r % 8)
// EG: fp32[128]: e^{Gamma_C}
constexpr uint32_t IMG_WQ = 0, IMG_KB = 32768, IMG_P = 49152, IMG_U = 57344;
__host__ __device__ constexpr uint32_t img_eg(int dv) { return IMG_U + 64u * dv * 2u; }
__host__ __device__ constexpr uint32_t img_bytes(int dv) { return img_eg(dv) + 512u; }

// ---- prep kernel shared memory ---------------------------------------------
constexpr int PNT = 256;                // prep threads: 64 channel pairs x 4 blocks of 16 tokens
constexpr uint32_t P_KHAT = 0;          // 16 KB  Khat K-major [64][128]; later T fp32 [64][68] (into APB)
constexpr uint32_t P_APB = 16384;       // 33 KB  [X; Y] K-major [128][128]; later A fp32 [64][65], XT
constexpr uint32_t P_KTIL = 50176;      // 16 KB  k e^{G} MN-major (mn = dk, K = 64)
constexpr uint32_t P_R1 = 66560;        // 32 KB  g tile; then [Khat_1; Khat_2; Khat_3]; then V + TOP
constexpr uint32_t P_KHS = P_R1;        // 24 KB  Khat_1, Khat_2, Khat_3 stacked: K-major [96][128]
constexpr uint32_t P_TOP = P_R1 + 16384;  // 16 KB [T; T] K-major [128][64]
constexpr uint32_t P_MISC = 99328;      // beta fp32[64] | mbar | tmem slot
constexpr uint32_t P_FAC = P_MISC + 512;  // bf16 [6][128]: e^{Gamma_m(R) - Gamma_m(S)}, S < R
constexpr uint32_t P_PART = P_FAC + 1536; // float4 [4][64]: per-block partial sums of g
constexpr uint32_t P_SMEM = P_PART + 4096 + 1024;

__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

constexpr float kLog2e = 1.4426950408889634f;
// 2^x with the hardware approximation (relative error ~2^-22); subnormal results
// are kept: a cross-block factor can be subnormal while its product with a
// large in-block factor is not
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// The same where the result is known to be normal: in-block factors
// e^{+-(Gamma_r - Gamma_m)} with |Gamma_r - Gamma_m| <= 8 |g_min| log2(e) < 126
// for g >= -10.
__device__ __forceinline__ float ex2_normal(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 u;
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  __nv_bfloat162 c = __floats2bfloat162_rn(v[4], v[5]), d = __floats2bfloat162_rn(v[6], v[7]);
  u.x = *reinterpret_cast<uint32_t*>(&a); u.y = *reinterpret_cast<uint32_t*>(&b);
  u.z = *reinterpret_cast<uint32_t*>(&c); u.w = *reinterpret_cast<uint32_t*>(&d);
  return u;
}

__device__ __forceinline__ int find_seq(const PrefillSched& s, int chunk) {
  int lo = 0, hi = s.n_seqs - 1;
  while (lo < hi) {                     // last n with chunk_base[n] <= chunk
    const int mid = (lo + hi + 1) >> 1;
    if (s.chunk_base[mid] <= chunk) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The CTA waits on an mbarrier: warp 0 polls it while the other warps sleep in
// the block barrier (no issue slots taken from the co-resident CTA); the barrier
// passes warp 0's acquire on to every thread and makes the outcome uniform.
__device__ __forceinline__ bool cta_wait(uint32_t mbar, uint32_t parity) {
  bool ok = true;
  if ((threadIdx.x >> 5) == 0) ok = mbar_wait(mbar, parity);
  return __syncthreads_and(ok) != 0;
}

// Tensor maps of one prefill launch: k and q as [T][H*128] with a 64 x 64 box
// and 128-byte swizzle (two boxes per chunk and head land as the K-major
// operand layout); g as [T][H*128] with a plain 128 x 64 box (row-major in
// shared memory); v as [T][H*DV] with a 64 x 64 box and 128-byte swizzle, which
// lands exactly in the MN-major operand layout the U = T V contraction reads.
struct PrepMaps {
  CUtensorMap k, q, g, v;
};

constexpr int TS = 68;                  // row stride of T in floats (16-byte rows)
constexpr uint32_t P_AF = P_APB + 1024;   // A fp32 [64][65] (T runs 1 KB into APB)
constexpr uint32_t P_XT = P_AF + 16640;   // intermediate products of the UT solve, fp32 [6][16][16]

template <int DV, bool DECAY_FIRST>
__global__ void __launch_bounds__(PNT, 2)
kda_chunk_prep_kernel(const PrefillArgs a, const PrefillSched sched, unsigned char* __restrict__ ws,
                      const __grid_constant__ PrepMaps maps) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  float* s_beta = reinterpret_cast<float*>(sm + P_MISC);
  const uint32_t mbar = smem_u32(sm + P_MISC + 256);       // tensor-core commits
  const uint32_t mbar_in = smem_u32(sm + P_MISC + 272);    // k, q and g tiles
  const uint32_t mbar_v = smem_u32(sm + P_MISC + 280);     // v tile
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + P_MISC + 264);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heads vary fastest across the grid: CTAs running together read whole token rows
  const int H = a.H;
  const int h = (int)(blockIdx.x % (unsigned)H), chunk = (int)(blockIdx.x / (unsigned)H);
  const int n = find_seq(sched, chunk);
  const int c = chunk - sched.chunk_base[n];
  const int64_t t0 = (int64_t)sched.start[n] + (int64_t)c * C;
  const int L = min(C, sched.len[n] - c * C);
  constexpr bool decay_first = DECAY_FIRST;
  unsigned char* img = ws + ((int64_t)chunk * H + h) * img_bytes(DV);
  const __nv_bfloat16* bg = reinterpret_cast<const __nv_bfloat16*>(a.beta);

  if (tid == 0) {
    // the chain launch that follows may start its CTAs once every prep CTA has
    // begun; it reads nothing of this grid before its grid-dependency wait
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    mbar_init(mbar, 1);
    mbar_init(mbar_in, 1);
    mbar_init(mbar_v, 1);
    mbar_init_fence();
    // k and q land 128-byte swizzled as the K-major rows 0-63 and 64-127 of the
    // [X; Y] operand, so the gating pass rewrites each element in place; the g
    // tile lands row-major in R1.
    mbar_expect_tx(mbar_in, 3 * 16384);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      tma_load_2d(smem_u32(sm + P_APB + b * 16384), &maps.k, h * DKT + 64 * b, (int)t0, mbar_in);
      tma_load_2d(smem_u32(sm + P_APB + b * 16384 + 8192), &maps.q, h * DKT + 64 * b, (int)t0, mbar_in);
    }
    tma_load_2d(smem_u32(sm + P_R1), &maps.g, h * DKT, (int)t0, mbar_in);
  }
  if (warp == 0) tmem_alloc(smem_u32(tslot), 256);
  if (tid < C) s_beta[tid] = tid < L ? ldf(bg + (t0 + tid) * H + h) : 0.f;
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  uint32_t phase = 0;
  bool ok = true;

  // ---- gates: thread t owns key channels 2p, 2p+1 (p = t % 64) for the 16
  // tokens of block qb = t / 64; every store is one packed bf16 pair.
  const int pch = tid & 63, qb = tid >> 6, c0 = 2 * pch;
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(sm + P_R1);   // g [64][64 pairs]
  float4* part = reinterpret_cast<float4*>(sm + P_PART);
  ok = cta_wait(mbar_in, 0);
  // Pass 1: sums of the block's 16 gates up to its reference token (the 8th)
  // and in total, exchanged so every thread has the cumsum at all four
  // reference tokens, at the end of the chunk and before its own block.  All
  // cumsums are kept in log2 units (g log2(e)), so every factor is one ex2.
  float2 gl[16];
  {
    // both channels in packed form: bf16 min / max of the gates (a NaN carries
    // through), packed fp32 scaling and sums (the roundings of scalar ones)
    const __nv_bfloat162 z2 = __float2bfloat162_rn(0.f);
    __nv_bfloat162 lo = z2, hi = z2;
    const float2 l2e = make_float2(kLog2e, kLog2e);
    float2 acc = make_float2(0.f, 0.f), half = acc;
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
      const int r = 16 * qb + rr;
      const __nv_bfloat162 graw = r < L ? g2[r * 64 + pch] : z2;
      lo = __hmin2_nan(lo, graw);
      hi = __hmax2_nan(hi, graw);
      gl[rr] = __fmul2_rn(__bfloat1622float2(graw), l2e);
      acc = __fadd2_rn(acc, gl[rr]);
      if (rr == 7) half = acc;
    }
    part[qb * 64 + pch] = make_float4(half.x, half.y, acc.x, acc.y);
    // the factor bounds below hold for g in [-10, 0]; anything else (or NaN)
    // raises the gate bit of the error word
    const float2 lof = __bfloat1622float2(lo), hif = __bfloat1622float2(hi);
    if (!(lof.x >= -10.f && lof.y >= -10.f && hif.x <= 0.f && hif.y <= 0.f))
      atomicOr(&g_kda_device_error, kDevErrGate);
  }
  __syncthreads();
  float gm[4][2], GC[2] = {0.f, 0.f}, acc0[2] = {0.f, 0.f};
#pragma unroll
  for (int R = 0; R < 4; ++R) {
    const float4 pr = part[R * 64 + pch];
    gm[R][0] = GC[0] + pr.x;
    gm[R][1] = GC[1] + pr.y;
    if (R < qb) { acc0[0] += pr.z; acc0[1] += pr.w; }
    GC[0] += pr.z;
    GC[1] += pr.w;
  }
  // block-to-block factors e^{Gamma_m(R) - Gamma_m(S)} <= 1 (S < R), six pairs
  __nv_bfloat162* fac2 = reinterpret_cast<__nv_bfloat162*>(sm + P_FAC);
  if (qb < 3) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int idx = 2 * qb + u;                       // (S, R) = (0,1) (0,2) (1,2) (0,3) (1,3) (2,3)
      const int R = idx == 0 ? 1 : (idx < 3 ? 2 : 3);
      const int S = idx - R * (R - 1) / 2;
      const float gR0 = R == 1 ? gm[1][0] : (R == 2 ? gm[2][0] : gm[3][0]);
      const float gR1 = R == 1 ? gm[1][1] : (R == 2 ? gm[2][1] : gm[3][1]);
      const float gS0 = S == 0 ? gm[0][0] : (S == 1 ? gm[1][0] : gm[2][0]);
      const float gS1 = S == 0 ? gm[0][1] : (S == 1 ? gm[1][1] : gm[2][1]);
      fac2[idx * 64 + pch] = __floats2bfloat162_rn(ex2(gR0 - gS0), ex2(gR1 - gS1));
    }
  } else {
    *reinterpret_cast<float2*>(img + img_eg(DV) + 4 * c0) = make_float2(ex2(GC[0]), ex2(GC[1]));
  }

  // Pass 2: every gated operand of the chunk for this thread's 16 tokens.  Row r
  // of Khat, k e^{G} and the image's Kbar share one offset (a [64][128] tile is
  // laid out alike K-major and MN-major), as do Y and the image's q e^{Gamma}.
  {
    const float gmq0 = qb == 0 ? gm[0][0] : (qb == 1 ? gm[1][0] : (qb == 2 ? gm[2][0] : gm[3][0]));
    const float gmq1 = qb == 0 ? gm[0][1] : (qb == 1 ? gm[1][1] : (qb == 2 ? gm[2][1] : gm[3][1]));
    const float em0 = ex2(gmq0), em1 = ex2(gmq1);                    // e^{Gamma_m}
    const float ec0 = ex2(GC[0] - gmq0), ec1 = ex2(GC[1] - gmq1);    // e^{Gamma_C - Gamma_m}
    // the two channels of a thread go through packed fp32 (two-lane) multiplies
    // and adds: the same roundings as scalar ones, half the instructions
    const float2 em = make_float2(em0, em1), ec = make_float2(ec0, ec1);
    auto rows = [&](auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;              // no token past the end
      float2 ac = make_float2(acc0[0] - gmq0, acc0[1] - gmq1);      // Gamma - Gamma_m, log2 units
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        const int r = 16 * qb + rr;
        const bool in = FULL || r < L;
        const uint32_t ox = off_k(r, c0, 128), oy = off_k(64 + r, c0, 128), o64 = off_k(r, c0, 64);
        __nv_bfloat162* xp = reinterpret_cast<__nv_bfloat162*>(sm + P_APB + ox);
        __nv_bfloat162* yp = reinterpret_cast<__nv_bfloat162*>(sm + P_APB + oy);
        const float2 kv = in ? __bfloat1622float2(*xp) : make_float2(0.f, 0.f);
        const float2 qv = in ? __bfloat1622float2(*yp) : make_float2(0.f, 0.f);
        const float2 p = ac;                        // Gamma_{r-1} - Gamma_m
        ac = __fadd2_rn(ac, gl[rr]);                // Gamma_r - Gamma_m
        const float2 E = make_float2(ex2_normal(ac.x), ex2_normal(ac.y));
        const float2 Ei = make_float2(ex2_normal(-ac.x), ex2_normal(-ac.y));
        const float2 EG = decay_first ? E : make_float2(ex2_normal(p.x), ex2_normal(p.y));
        const float2 Fq = __fmul2_rn(E, em);        // e^{Gamma}
        const float2 Fg = __fmul2_rn(EG, em);       // e^{G}
        const float2 Fc = __fmul2_rn(Ei, ec);       // e^{Gamma_C - Gamma}
        *reinterpret_cast<__nv_bfloat162*>(sm + P_KHAT + o64) = __float22bfloat162_rn(__fmul2_rn(kv, Ei));
        *reinterpret_cast<__nv_bfloat162*>(sm + P_KTIL + o64) = __float22bfloat162_rn(__fmul2_rn(kv, Fg));
        *reinterpret_cast<__nv_bfloat162*>(img + IMG_WQ + oy) = __float22bfloat162_rn(__fmul2_rn(qv, Fq));
        *reinterpret_cast<__nv_bfloat162*>(img + IMG_KB + o64) = __float22bfloat162_rn(__fmul2_rn(kv, Fc));
        *xp = __float22bfloat162_rn(__fmul2_rn(kv, EG));     // X = k e^{G - Gamma_m}
        *yp = __float22bfloat162_rn(__fmul2_rn(qv, E));      // Y = q e^{Gamma - Gamma_m}
      }
    };
    if (L == C) rows(std::true_type{}); else rows(std::false_type{});
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();

  // ---- A and P on tcgen05: D = [X; Y] x (K side)^T over all 128 rows --------
  // Row block R takes its factor split at reference token m(R): the diagonal
  // block reads Khat (k e^{Gamma_m(R) - Gamma}) as it is; the blocks left of it
  // read Khat_R = Khat x e^{Gamma_m(R) - Gamma_m(S)}, built once per R.
  // Two products: [X; Y] x Khat^T into TMEM columns 0-63 (row block R keeps
  // columns 16 R .. 16 R + 15, its diagonal block) and [X; Y] x [Khat_1; Khat_2;
  // Khat_3]^T into columns 64-159 (Khat_1 at 64, Khat_2 at 80, Khat_3 at 112).
  const uint32_t apb = smem_u32(sm + P_APB);
  const uint32_t khat = smem_u32(sm + P_KHAT);
  if (ok && warp == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      mma_w(tmem, desc_k(apb, 128, j), desc_k(khat, 64, j), idesc_bf16(128, 64, false, false), j > 0);
  }
  {
    const __nv_bfloat16* facb = reinterpret_cast<const __nv_bfloat16*>(sm + P_FAC);
    const int sr = tid >> 4, cc = tid & 15;
#pragma unroll
    for (int m = 0; m < 6; ++m) {
      const int R = m == 0 ? 1 : (m < 3 ? 2 : 3);
      const int S = m == 0 ? 0 : (m < 3 ? m - 1 : m - 3);
      const int s = 16 * S + sr;
      const int row0 = R == 1 ? 0 : (R == 2 ? 16 : 48);            // Khat_R's first row in the stack
      const uint4 x = *reinterpret_cast<const uint4*>(sm + P_KHAT + off_k(s, 8 * cc, 64));
      const uint4 f = *reinterpret_cast<const uint4*>(facb + (R * (R - 1) / 2 + S) * DKT + 8 * cc);
      uint4 y;
      const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&x);
      const __nv_bfloat162* fp = reinterpret_cast<const __nv_bfloat162*>(&f);
      __nv_bfloat162* yp = reinterpret_cast<__nv_bfloat162*>(&y);
#pragma unroll
      for (int t = 0; t < 4; ++t) yp[t] = __hmul2(xp[t], fp[t]);
      *reinterpret_cast<uint4*>(sm + P_KHS + off_k(row0 + s, 8 * cc, 96)) = y;
    }
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();
  if (ok && warp == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      mma_w(tmem + 64, desc_k(apb, 128, j), desc_k(smem_u32(sm + P_KHS), 96, j), idesc_bf16(128, 96, false, false),
            j > 0);
    mma_commit_w(mbar);
  }
  if (ok) { ok = cta_wait(mbar, phase); phase ^= 1; fence_after(); }
  // the A/P products are done with the stacked Khat_R: v lands there (MN-major,
  // swizzled), right after k e^{G}, so [k e^{G} | v] is one B operand
  const bool v_issued = ok;
  if (ok && tid == 0) {
    mbar_expect_tx(mbar_v, 64 * DV * 2);
#pragma unroll
    for (int b = 0; b < DV / 64; ++b)
      tma_load_2d(smem_u32(sm + P_R1 + b * 8192), &maps.v, h * DV + 64 * b, (int)t0, mbar_v);
  }

  // ---- read A (lanes 0-63) and P (lanes 64-127); warps w and w + 4 share a
  // lane quadrant and take the left and right columns of its rows.
  float* AF = reinterpret_cast<float*>(sm + P_AF);             // [64][65]
  float* TF = reinterpret_cast<float*>(sm + P_KHAT);           // [64][TS]
  if (ok) {
    const int qd = warp & 3, hw = warp >> 2;
    const bool lo = lane < 16;
    const int r = 32 * (qd & 1) + lane;                         // token row of this lane
    const uint32_t la = tmem + ((uint32_t)(32 * qd) << 16);
    float v[32];
    int s0, nv;                                                 // v holds columns s0 .. s0 + nv - 1
    if ((qd & 1) == 0) {                                        // rows 0-31: blocks 0 and 1
      float a16[16];
      if (hw == 0) {
        float b16[16];
        tmem_ld16(la + 0, a16);
        tmem_ld16(la + 64, b16);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = lo ? a16[e] : b16[e];
        s0 = 0;
      } else {
        tmem_ld16(la + 16, a16);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = a16[e];
        s0 = 16;
      }
#pragma unroll
      for (int e = 16; e < 32; ++e) v[e] = 0.f;
      nv = 16;
    } else {                                                    // rows 32-63: blocks 2 and 3
      if (hw == 0) {
        float b[32];
        tmem_ld32(la + 80, v);
        tmem_ld32(la + 112, b);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = lo ? v[e] : b[e];
        s0 = 0;
      } else {
        float b16[16];
        tmem_ld32(la + 32, v);
        tmem_ld16(la + 144, b16);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = lo ? v[e] : b16[e];
        s0 = 32;
      }
      nv = 32;
    }
    if (qd < 2) {
      // entries with s >= r are never read; two columns per packed fp32 multiply
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        if (e < nv) {
          const int s = s0 + e;
          const float2 b2 = *reinterpret_cast<const float2*>(s_beta + s);
          const float2 x = __fmul2_rn(make_float2(v[e], v[e + 1]), b2);
          AF[r * 65 + s] = x.x;
          AF[r * 65 + s + 1] = x.y;
        }
      }
    } else {
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        if (8 * q8 < nv) {
          float p8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) p8[e] = s0 + 8 * q8 + e <= r ? v[8 * q8 + e] : 0.f;
          *reinterpret_cast<uint4*>(img + IMG_P + off_k(r, s0 + 8 * q8, 64)) = pack8(p8);
        }
      }
      if ((qd & 1) == 0 && hw == 1) {                           // rows 0-31 are zero right of column 31
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8)
          *reinterpret_cast<uint4*>(img + IMG_P + off_k(r, 32 + 8 * q8, 64)) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  // (T's blocks above the diagonal are never stored: the [T; T] build writes their zeros)
  fence_before();
  __syncthreads();
  fence_after();

  // ---- UT solve T = (I + A)^{-1}: 16x16 diagonal blocks, then block levels --
  if (tid < 64) {
    // column cc of the inverse of diagonal block J, by forward substitution
    const int J = tid >> 4, cc = tid & 15, b0 = 16 * J;
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float arow[16];
#pragma unroll
      for (int s2 = 0; s2 < j; ++s2) arow[s2] = AF[(b0 + j) * 65 + b0 + s2];
      // even and odd terms in the two lanes of one packed fp32 accumulator
      float2 e = make_float2(0.f, 0.f);
#pragma unroll
      for (int s2 = 0; s2 + 1 < j; s2 += 2)
        e = __ffma2_rn(make_float2(arow[s2], arow[s2 + 1]), make_float2(x[s2], x[s2 + 1]), e);
      if (j & 1) e.x = fmaf(arow[j - 1], x[j - 1], e.x);
      x[j] = j == cc ? 1.f : (j < cc ? 0.f : -(e.x + e.y));
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) TF[(b0 + j) * TS + b0 + cc] = x[j];
  }
  __syncthreads();
  // Off-diagonal blocks by 2x2 doubling: T = [[T1, 0], [-T2 A21 T1, T2]] on the
  // 32x32 halves, whose own off-diagonal blocks come first the same way.
  // XT slots [6][16][16]: 0 A10 T00, 1 A32 T22, 2 A21 T11, 3 A31 T11, 4 A20 T00
  // (+ A21 T10), 5 A30 T00 (+ A31 T10).  One thread per row and 4 columns.
  float* XT = reinterpret_cast<float*>(sm + P_XT);
  // the strip's four columns as two packed fp32 fused multiply-adds (fmaf's rounding)
  auto fma4 = [](float a, float4 b, float4 acc) {
    const float2 aa = make_float2(a, a);
    const float2 lo = __ffma2_rn(aa, make_float2(b.x, b.y), make_float2(acc.x, acc.y));
    const float2 hi = __ffma2_rn(aa, make_float2(b.z, b.w), make_float2(acc.z, acc.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  };
  auto a_t = [&](int I, int K, int J, int ar, int bq, float4 acc) {   // acc += A_IK T_KJ (row ar, cols 4bq..)
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2) {
      const float av = AF[(16 * I + ar) * 65 + 16 * K + s2];
      acc = fma4(av, *reinterpret_cast<const float4*>(TF + (16 * K + s2) * TS + 16 * J + 4 * bq), acc);
    }
    return acc;
  };
  auto t_x = [&](int I, int L, int slot, int ar, int bq, bool tri, float4 acc) {   // acc += T_IL X_slot
#pragma unroll
    for (int s2 = 0; s2 < 16; ++s2) {
      if (!tri || s2 <= ar) {
        const float tv = TF[(16 * I + ar) * TS + 16 * L + s2];
        acc = fma4(tv, *reinterpret_cast<const float4*>(XT + slot * 256 + s2 * 16 + 4 * bq), acc);
      }
    }
    return acc;
  };
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const int ar = (tid >> 2) & 15, bq = tid & 3, blk = tid >> 6;
  auto put = [&](float* base, float4 v) { *reinterpret_cast<float4*>(base) = v; };
  auto neg = [](float4 v) { return make_float4(-v.x, -v.y, -v.z, -v.w); };
  // 1: products of A with diagonal blocks only (six blocks, two per thread for tid < 128)
  {
    const int I1[4] = {1, 3, 2, 3}, K1[4] = {0, 2, 1, 1}, J1[4] = {0, 2, 1, 1};
    float4 r = z4;
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (blk == b) r = a_t(I1[b], K1[b], J1[b], ar, bq, z4);
    put(XT + blk * 256 + ar * 16 + 4 * bq, r);
    if (tid < 128) {
      const int I = blk == 0 ? 2 : 3;                        // slots 4 and 5: A20 T00, A30 T00
      put(XT + (4 + blk) * 256 + ar * 16 + 4 * bq, a_t(I, 0, 0, ar, bq, z4));
    }
  }
  __syncthreads();
  // 2: T10 = -T11 (A10 T00), T32 = -T33 (A32 T22)
  if (tid < 128) {
    const int I = blk == 0 ? 1 : 3, J = I - 1;
    put(TF + (16 * I + ar) * TS + 16 * J + 4 * bq, neg(t_x(I, I, blk, ar, bq, true, z4)));
  }
  __syncthreads();
  // 3: slots 4, 5 += A21 T10, A31 T10
  if (tid < 128) {
    const int I = blk == 0 ? 2 : 3;
    float* xp = XT + (4 + blk) * 256 + ar * 16 + 4 * bq;
    put(xp, a_t(I, 1, 0, ar, bq, *reinterpret_cast<const float4*>(xp)));
  }
  __syncthreads();
  // 4: T20 = -T22 X20, T21 = -T22 X21, T30 = -(T32 X20 + T33 X30), T31 = -(T32 X21 + T33 X31)
  {
    const int I = blk < 2 ? 2 : 3, J = blk & 1;
    const int sx2 = J == 0 ? 4 : 2, sx3 = J == 0 ? 5 : 3;   // X_2J and X_3J slots
    float4 r;
    if (I == 2) {
      r = t_x(2, 2, sx2, ar, bq, true, z4);
    } else {
      r = t_x(3, 2, sx2, ar, bq, false, z4);
      r = t_x(3, 3, sx3, ar, bq, true, r);
    }
    put(TF + (16 * I + ar) * TS + 16 * J + 4 * bq, neg(r));
  }
  __syncthreads();

  // ---- [T; T] as bf16 A operand (the copy feeds lanes 64-127) -----------------
  {
    const int r = tid & 127, c32 = 32 * (tid >> 7);
#pragma unroll
    for (int cch = 0; cch < 4; ++cch) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);              // zero above the diagonal blocks
      if ((c32 + 8 * cch) >> 4 <= (r & 63) >> 4) {
        const float4 lo = *reinterpret_cast<const float4*>(TF + (r & 63) * TS + c32 + 8 * cch);
        const float4 hi = *reinterpret_cast<const float4*>(TF + (r & 63) * TS + c32 + 8 * cch + 4);
        const float t8[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        w = pack8(t8);
      }
      *reinterpret_cast<uint4*>(sm + P_TOP + off_k(r, c32 + 8 * cch, 128)) = w;
    }
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();
  if (ok) ok = cta_wait(mbar_v, 0);     // v rows past the sequence end meet beta = 0
  if (ok && warp == 0) {
    const uint32_t top = smem_u32(sm + P_TOP);
    constexpr uint32_t ID_WU = idesc_bf16(128, 128 + DV, false, true);   // W in columns 0-127, U after
#pragma unroll
    for (int j = 0; j < 4; ++j) mma_w(tmem, desc_k(top, 128, j), desc_mn(smem_u32(sm + P_KTIL), 64, j), ID_WU, j > 0);
    mma_commit_w(mbar);
  }
  if (ok) { ok = cta_wait(mbar, phase); phase ^= 1; fence_after(); }

  // ---- -beta W (lanes 0-63) and beta U (lanes 64-127) to the chunk image -----
  if (ok) {
    const int qd = warp & 3, hw = warp >> 2;
    const int r = (32 * qd + lane) & 63;
    const uint32_t la = tmem + ((uint32_t)(32 * qd) << 16);
    const float br = s_beta[r];
    if (qd < 2) {
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        const int j = 64 * hw + 16 * cb;
        float v[16];
        tmem_ld16(la + j, v);
        const float2 nb = make_float2(-br, -br);
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float2 x = __fmul2_rn(make_float2(v[e], v[e + 1]), nb);
          v[e] = x.x;
          v[e + 1] = x.y;
        }
        *reinterpret_cast<uint4*>(img + IMG_WQ + off_k(r, j, 128)) = pack8(v);
        *reinterpret_cast<uint4*>(img + IMG_WQ + off_k(r, j + 8, 128)) = pack8(v + 8);
      }
    } else {
#pragma unroll
      for (int cb = 0; cb < DV / 32; ++cb) {
        const int j = (DV / 2) * hw + 16 * cb;
        float v[16];
        tmem_ld16(la + 128 + j, v);
        const float2 pb = make_float2(br, br);
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float2 x = __fmul2_rn(make_float2(v[e], v[e + 1]), pb);
          v[e] = x.x;
          v[e + 1] = x.y;
        }
        // row r of each 64-column block: 16-byte chunk c at position c ^ (r % 8), so the
        // chain's row-per-thread reads hit distinct banks
        unsigned char* blk = img + IMG_U + (j >> 6) * 8192 + r * 128;
        const int cj = (j & 63) >> 3;
        *reinterpret_cast<uint4*>(blk + (((cj) ^ (r & 7)) << 4)) = pack8(v);
        *reinterpret_cast<uint4*>(blk + (((cj + 1) ^ (r & 7)) << 4)) = pack8(v + 8);
      }
    }
  }
  if (!ok && tid == 0) {
    // leave no bulk copy in flight into this CTA's shared memory (bounded waits)
    mbar_wait(mbar_in, 0);
    if (v_issued) mbar_wait(mbar_v, 0);
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---- chain kernel -------------------------------------------------------------
// One CTA per (sequence, head, slice of DVS = 32 or 64 columns of dv), ten
// warps: 32-column slices when 64-column ones would leave more than half of
// the SMs idle (the chain is latency-bound, and an N = 32 product reads 5 KB
// of operands instead of 6 KB while the per-row register work halves).  Warps
// 0-7 own the state rows, warps w and w + 4 sharing TMEM lane quadrant w % 4
// and taking the left and right DVS / 2 columns of its rows; warp 8 writes
// checkpoint pages from a staging buffer the row warps fill, so no global
// store precedes a hand-off on the critical path; warp 9 streams the chunk
// images into a two-stage ring.  Each product is issued by warp 0 right after
// a named barrier of the warps that wrote its operand: Kbar^T Delta' (MMA3)
// and P Delta' (MMA2) after the four Delta' warps (0, 1, 4, 5), [-bW; Qt] S
// (MMA1) of the next chunk after all eight row warps have staged the state.
// The output rows of a chunk are read back by warps 2, 3, 6, 7 while the next
// chunk's Delta' is formed, when the tensor pipe is idle and they would only
// wait.  Products report completion on mbarriers (bar1, bar3, bar2).  A ring
// stage goes back to warp 9 after nine arrivals: the commit issued after MMA2
// (every product reading the stage is then done) and one per row warp after
// its last read of the stage, at the top of the step.
// Both named barriers OR an error flag over their warps, so the row warps
// leave the loop together; every mbarrier wait is bounded and watches the
// abort flag.
constexpr int CNT = 320;                           // chain threads: 8 row warps, writer, producer
constexpr int PRODUCER = 9;                        // the image-copy warp
constexpr int CRW = 256;                           // row threads
constexpr uint32_t S_WQ = 0, S_KB = 32768, S_PB = 49152, S_U = 65536, S_EG = 73728;
constexpr uint32_t STAGE = 75776;                 // 74 KB, keeps every stage 1024-aligned
constexpr uint32_t C_DELTA = 2 * STAGE;           // 8 KB  Delta' MN-major (mn = DVS cols, K = 64 tokens)
constexpr uint32_t C_SB = C_DELTA + 8192;         // 16 KB S bf16 MN-major (mn = DVS cols, K = 128)
constexpr uint32_t C_MISC = C_SB + 16384;
constexpr uint32_t C_CK = C_MISC + 128;           // 34 KB checkpoint staging: fp32 [128 rows][DVS], rows 272 B apart
constexpr uint32_t CK_ROW = 272;
constexpr uint32_t C_SMEM = C_CK + 128 * CK_ROW + 1024;
constexpr uint32_t CHUNK_TX = 32768 + 16384 + 8192 + 8192 + 512;

// TMEM -> registers, 16 or 32 consecutive columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[16]) { tmem_ld16(taddr, v); }
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[32]) { tmem_ld32(taddr, v); }

// Named barrier over `nthreads` threads that also ORs a predicate over them:
// every participant gets the same answer.
__device__ __forceinline__ bool bar_sync_or(int id, int nthreads, bool pred) {
  int r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.s32 p, %1, 0; barrier.cta.red.or.pred q, %2, %3, p; selp.s32 %0, 1, 0, q; }"
      : "=r"(r) : "r"((int)pred), "r"(id), "r"(nthreads) : "memory");
  return r != 0;
}
// A whole warp waits on an mbarrier phase (bounded, abort-aware); the result is warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t mbar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_test(mbar, parity) || mbar_wait_or_abort(mbar, parity, abort_flag));
}

template <int DV, int DVS>
__global__ void __launch_bounds__(CNT, 1)
kda_chain_kernel(const PrefillArgs a, const PrefillSched sched, const unsigned char* __restrict__ ws) {
  static_assert(DVS == 32 || DVS == 64, "a chain CTA owns 32 or 64 state columns");
  constexpr int NC = DVS / 2;                          // state columns per row thread
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t full0 = smem_u32(sm + C_MISC);         // two image stages landed
  const uint32_t bar1 = smem_u32(sm + C_MISC + 16);     // [-bW; Qt] S done
  const uint32_t bar3 = smem_u32(sm + C_MISC + 24);     // Kbar^T Delta' done
  const uint32_t bar2 = smem_u32(sm + C_MISC + 32);     // P Delta' done
  const uint32_t free0 = smem_u32(sm + C_MISC + 40);    // two image stages released
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C_MISC + 64);
  const uint32_t ckfull = smem_u32(sm + C_MISC + 88);   // staging filled (8 row warps)
  const uint32_t ckfree = smem_u32(sm + C_MISC + 96);   // staging written out (warp 8)
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + C_MISC + 72);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, hh = (warp >> 2) & 1;       // lane quadrant, column half (row warps)
  const int sl = blockIdx.x, h = blockIdx.y, H = a.H;
  const int n = sched.order[blockIdx.z];
  const int64_t start = sched.start[n];
  const int len = sched.len[n];
  const int nch = (len + C - 1) / C;
  const int64_t ib = img_bytes(DV);
  const unsigned char* img0 = ws + ((int64_t)sched.chunk_base[n] * H + h) * ib;
  const int col0 = sl * DVS;
  const int jc = NC * hh;                              // this thread's first column inside the slice

  if (tid == 0) {
    mbar_init(full0, 1);
    mbar_init(full0 + 8, 1);
    mbar_init(bar1, 1);
    mbar_init(bar3, 1);
    mbar_init(bar2, 1);
    mbar_init(free0, 9);                 // the products' commit and the eight row warps
    mbar_init(free0 + 8, 9);
    mbar_init(ckfull, 8);
    mbar_init(ckfree, 1);
    *s_abort = 0;
    mbar_init_fence();
  }
  if (warp == PRODUCER) tmem_alloc(smem_u32(tslot), 256);
  // launched as a programmatic dependent of the preceding kernel (the prep, or the
  // scan kernel that makes S0): everything below may read what it wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // zero rows 0-63 of both [0; P] buffers (never written by the copies)
  for (int e = tid; e < 2 * 512; e += CNT) {
    const int s = e >> 9, o = e & 511;
    reinterpret_cast<uint4*>(sm + s * STAGE + S_PB)[o] = make_uint4(0, 0, 0, 0);
  }
  // row warps: state row i, columns col0 + jc .. col0 + jc + NC - 1
  const int i = 32 * qd + lane;
  float S[NC];
  if (warp < 8) {
    const int64_t srow = (((int64_t)n * H + h) * DKT + i) * DV + col0 + jc;
#pragma unroll
    for (int j = 0; j < NC; j += 4) {
      float4 x = a.S0 ? *reinterpret_cast<const float4*>(a.S0 + srow + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
    }
#pragma unroll
    for (int cch = 0; cch < NC / 8; ++cch)
      *reinterpret_cast<uint4*>(sm + C_SB + off_mn(jc + 8 * cch, i, 128)) = pack8(S + 8 * cch);
  }
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  // TMEM: two output/WS accumulators (one per chunk parity) and the state update
  const uint32_t d2 = tmem + 128;          // d1 of chunk c: tmem + 64 * (c & 1)
  const uint32_t delta = smem_u32(sm + C_DELTA), sb = smem_u32(sm + C_SB);
  constexpr uint32_t ID_1 = idesc_bf16(128, DVS, false, true);   // [-bW; Qt] (K-major) x S (MN-major)
  constexpr uint32_t ID_3 = idesc_bf16(128, DVS, true, true);    // Kbar^T (MN-major) x Delta' (MN-major)

  if (warp == PRODUCER) {
    // ---- image copies: stage c & 1 of chunk c, once the products of chunk c - 2
    // are complete and the row warps are through it (the free commit) ----------
    if (lane == 0) {
      auto copy = [&](int cidx) {
        const int s = cidx & 1;
        const unsigned char* src = img0 + (int64_t)cidx * H * ib;
        const uint32_t dst = smem_u32(sm + s * STAGE);
        const uint32_t fb = full0 + 8 * s;
        mbar_expect_tx(fb, CHUNK_TX);
        bulk_g2s(dst + S_WQ, src + IMG_WQ, 32768, fb);
        bulk_g2s(dst + S_KB, src + IMG_KB, 16384, fb);
        bulk_g2s(dst + S_PB + 8192, src + IMG_P, 8192, fb);
        bulk_g2s(dst + S_U, src + IMG_U + (col0 >> 6) * 8192, 8192, fb);   // the 64-column block of the slice
        bulk_g2s(dst + S_EG, src + img_eg(DV), 512, fb);
      };
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        if (c >= 2 && !mbar_wait_or_abort(free0 + 8 * (c & 1), (uint32_t)(((c - 2) >> 1) & 1), s_abort)) {
          *s_abort = 1;
          break;
        }
        copy(c);
        issued = c + 1;
      }
      // leave no copy in flight into this CTA's shared memory (bounded waits; a
      // phase that already completed returns at once)
      for (int cc = max(0, issued - 2); cc < issued; ++cc) mbar_wait(full0 + 8 * (cc & 1), (uint32_t)((cc >> 1) & 1));
    }
    __syncwarp();
  } else if (warp == 8) {
    // ---- checkpoint writer: each staged checkpoint, 128 rows of 256 bytes --------
    const int ck_every = a.ckpt_stride > 0 && (sched.flags[n] & kSeqEmit) ? a.ckpt_stride / C : 0;
    int k = 0;
    if (ck_every > 0) {
      for (int c = ck_every - 1; c < nch; c += ck_every) {
        const int L = min(C, len - c * C);
        if (L != C) break;
        const int64_t idx = (int64_t)sched.ckpt_base[n] + (c * C + L) / a.ckpt_stride - 1;
        if (idx >= a.num_ckpt) break;
        const int32_t page_id = a.ckpt_page_ids[idx];
        // one bounded wait: it ends when the rows are staged, when another warp
        // aborts, or after about a second (error word raised); either failure
        // ends this warp's loop and aborts the CTA
        if (!warp_wait(ckfull, (uint32_t)(k & 1), s_abort)) {
          *s_abort = 1;
          break;
        }
        char* page = a.page_pool + (int64_t)page_id * a.page_bytes;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int row = lane + 32 * q4;
          bulk_s2g(page + (((int64_t)h * DKT + row) * DV + col0) * 4, smem_u32(sm + C_CK + row * CK_ROW), DVS * 4);
        }
        bulk_commit();
        bulk_wait_read_all();
        __syncwarp();
        if (lane == 0) mbar_arrive(ckfree);
        ++k;
      }
    }
    bulk_wait_all();
  } else {
    // ---- row warps -------------------------------------------------------------
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.o);
    const uint32_t lane_off = (uint32_t)(32 * qd) << 16;
    const bool emit = (sched.flags[n] & kSeqEmit) != 0, use_u = (sched.flags[n] & kSeqNoU) == 0;
    const int ck_every = a.ckpt_stride > 0 && emit ? a.ckpt_stride / C : 0;
    int ck_left = ck_every;
    int n_ck = 0;                          // checkpoints staged so far
    // operand descriptors, computed once: k-step j only moves the start address
    // (16-byte units in the low bits): +2 j within a 128-byte swizzle row and
    // +8 * R per 64-element K block (K-major, R rows), +128 j (MN-major)
    const uint64_t dS = desc_mn(sb, 128, 0), dD = desc_mn(delta, 64, 0);
    const uint64_t dW0 = desc_k(smem_u32(sm + S_WQ), 128, 0), dW1 = desc_k(smem_u32(sm + STAGE + S_WQ), 128, 0);
    const uint64_t dK0 = desc_mn(smem_u32(sm + S_KB), 64, 0), dK1 = desc_mn(smem_u32(sm + STAGE + S_KB), 64, 0);
    const uint64_t dP0 = desc_k(smem_u32(sm + S_PB), 128, 0), dP1 = desc_k(smem_u32(sm + STAGE + S_PB), 128, 0);
    // products issued by warp 0 (all lanes run these; one elected lane issues)
    int last1 = -1, last32 = -1;           // last chunk whose MMA1 / MMA3+MMA2 were issued (warp 0)
    auto mma1 = [&](auto stage_tag, int cidx) {
      constexpr int s = decltype(stage_tag)::value;
      const uint64_t dW = s ? dW1 : dW0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        mma_w(tmem + 64u * s, dW + (uint64_t)((j >> 2) * 1024 + (j & 3) * 2), dS + (uint64_t)(128 * j), ID_1, j > 0);
      mma_commit_w(bar1);
      last1 = cidx;
    };
    auto mma32 = [&](auto stage_tag, int cidx) {
      constexpr int s = decltype(stage_tag)::value;
      const uint64_t dK = s ? dK1 : dK0, dP = s ? dP1 : dP0;
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_w(d2, dK + (uint64_t)(128 * j), dD + (uint64_t)(128 * j), ID_3, j > 0);
      mma_commit_w(bar3);
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_w(tmem + 64u * s, dP + (uint64_t)(2 * j), dD + (uint64_t)(128 * j), ID_1, 1);
      mma_commit_w(bar2);
      // every product reading this stage is issued: their completion is the first
      // release arrival of the stage (the row warps give the other eight)
      mma_commit_w(free0 + 8 * s);
      last32 = cidx;
    };
    // outputs of chunk cc: rows 64-127 of d1[cc & 1] (warps 2, 3, 6, 7); the buffer is
    // next written by chunk cc + 2's MMA1, issued after these warps pass chunk cc + 1's
    // eight-warp barrier.  Chunk cc's MMA2 is known complete once chunk cc + 1's bar1
    // has been seen (warp 0 commits that after issuing the MMA2); only the last
    // chunk waits on bar2 itself.
    auto read_outputs = [&](int cc, bool wait_bar2) -> bool {
      if (wait_bar2 && !warp_wait(bar2, (uint32_t)(cc & 1), s_abort)) return false;
      fence_after();
      float ov[NC];
      tmem_ld_cols(tmem + 64u * (cc & 1) + lane_off + jc, ov);
      const int r = i - 64;
      if (emit && r < min(C, len - cc * C)) {
        __nv_bfloat16* orow = o + ((start + (int64_t)cc * C + r) * H + h) * DV + col0 + jc;
#pragma unroll
        for (int q8 = 0; q8 < NC / 8; ++q8) *reinterpret_cast<uint4*>(orow + 8 * q8) = pack8(ov + 8 * q8);
      }
      return true;
    };
    if (nch > 0 && warp == 0) {
      if (warp_wait(full0, 0, s_abort)) {
        fence_after();
        mma1(std::integral_constant<int, 0>{}, 0);
      } else {
        *s_abort = 1;
      }
    }
    auto row_step = [&](auto stage_tag, int c) -> bool {
      constexpr int s = decltype(stage_tag)::value;
      const uint32_t ph = (uint32_t)(c & 1);
      const unsigned char* st = sm + s * STAGE;
      const uint32_t d1 = tmem + 64u * s;
      // the images of chunk c (landed long ago; acquires them for this thread)
      bool good = warp_wait(full0 + 8 * s, (uint32_t)((c >> 1) & 1), s_abort);
      // shared-memory inputs of this chunk's row work, loaded before the waits
      // on the products
      const float eg = good ? reinterpret_cast<const float*>(st + S_EG)[i] : 0.f;
      // this warp's last read of the stage: its release arrival, so the copy of
      // chunk c + 2 can start once the products are done as well
      auto release = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(free0 + 8 * s);
      };
      if (qd < 2) {                         // Delta' = beta U - beta W S, token row r
        const int r = i;
        const uint4* urow = reinterpret_cast<const uint4*>(st + S_U + r * 128);
        const int cb0 = ((col0 & 63) + jc) >> 3;             // first 16-byte chunk of this thread's columns
        uint4 u[NC / 8];
#pragma unroll
        for (int cc = 0; cc < NC / 8; ++cc)
          u[cc] = good && use_u ? urow[(cb0 + cc) ^ (r & 7)] : make_uint4(0u, 0u, 0u, 0u);
        release();
        good = good && warp_wait(bar1, ph, s_abort);
        if (good) {
          fence_after();
          float v[NC];
          tmem_ld_cols(d1 + lane_off + jc, v);
#pragma unroll
          for (int cc = 0; cc < NC / 8; ++cc) {
            const __nv_bfloat162* pu = reinterpret_cast<const __nv_bfloat162*>(&u[cc]);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float2 x = __bfloat1622float2(pu[t]);
              v[8 * cc + 2 * t] += x.x;
              v[8 * cc + 2 * t + 1] += x.y;
            }
          }
#pragma unroll
          for (int cc = 0; cc < NC / 8; ++cc)
            *reinterpret_cast<uint4*>(sm + C_DELTA + off_mn(jc + 8 * cc, r, 64)) = pack8(v + 8 * cc);
          fence_async_smem();
        }
        fence_before();
        if (bar_sync_or(1, 128, !good)) {     // the four Delta' warps
          *s_abort = 1;
          good = false;
        } else if (warp == 0) {
          fence_after();
          mma32(stage_tag, c);
        }
      } else {
        release();
        // the previous chunk's outputs, read while Delta' is formed: this chunk's
        // MMA1 is complete first, so the tensor pipe is idle meanwhile
        if (c > 0) good = good && warp_wait(bar1, ph, s_abort) && read_outputs(c - 1, false);
      }
      // state update: S_i <- e^{Gamma_C,i} S_i + (Kbar^T Delta')_i
      good = good && warp_wait(bar3, ph, s_abort);
      if (good) {
        fence_after();
        float v[NC];
        tmem_ld_cols(d2 + lane_off + jc, v);
#pragma unroll
        for (int j = 0; j < NC; ++j) S[j] = fmaf(eg, S[j], v[j]);
#pragma unroll
        for (int cch = 0; cch < NC / 8; ++cch)
          *reinterpret_cast<uint4*>(sm + C_SB + off_mn(jc + 8 * cch, i, 128)) = pack8(S + 8 * cch);
      }
      const int L = min(C, len - c * C);
      const int pos = c * C + L;
      // a checkpoint ends every ckpt_stride / C full chunks (a partial chunk
      // never ends on a multiple of the stride); its rows go to the staging
      // buffer once warp 8 has written out the previous checkpoint
      const bool ck = ck_every > 0 && --ck_left == 0;
      if (ck) ck_left = ck_every;
      if (good && ck && L == C) {
        const int64_t idx = (int64_t)sched.ckpt_base[n] + pos / a.ckpt_stride - 1;
        if (idx < a.num_ckpt) {
          good = n_ck == 0 || warp_wait(ckfree, (uint32_t)((n_ck - 1) & 1), s_abort);
          if (good) {
            float4* srow = reinterpret_cast<float4*>(sm + C_CK + i * CK_ROW + jc * 4);
#pragma unroll
            for (int j = 0; j < NC / 4; ++j) srow[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ckfull);
            ++n_ck;
            if (h == 0 && sl == 0) {
              float* page = reinterpret_cast<float*>(a.page_pool + (int64_t)a.ckpt_page_ids[idx] * a.page_bytes);
              const int64_t used = (int64_t)H * DKT * DV, total = a.page_bytes / 4;
              for (int64_t e = used + tid; e < total; e += CRW) page[e] = 0.f;   // pad past the state
              if (tid == 0 && a.ckpt_pos) a.ckpt_pos[idx] = sched.pos_base[n] + pos;
            }
          }
        }
      }
      fence_async_smem();
      fence_before();
      if (bar_sync_or(2, CRW, !good)) {       // all eight row warps
        *s_abort = 1;
        return false;
      }
      if (warp == 0) {
        fence_after();
        // the next chunk's MMA1
        if (c + 1 < nch) {
          if (warp_wait(full0 + 8 * (s ^ 1), (uint32_t)(((c + 1) >> 1) & 1), s_abort)) {
            fence_after();
            mma1(std::integral_constant<int, s ^ 1>{}, c + 1);
          } else {
            *s_abort = 1;                   // the other warps see it at their next wait
          }
        }
      }
      return true;
    };
    int c = 0;
    // warp 0's failure before the loop reaches the other warps through the abort
    // flag at their first wait, and every warp then leaves at the first barrier
    bool ok = true;
    while (c < nch) {
      if (!(ok = row_step(std::integral_constant<int, 0>{}, c)) || ++c >= nch) break;
      if (!(ok = row_step(std::integral_constant<int, 1>{}, c))) break;
      ++c;
    }
    // the last chunk's outputs (no later chunk reads them back)
    if (ok && nch > 0 && qd >= 2 && !read_outputs(nch - 1, true)) *s_abort = 1;
    if (warp == 0 && *s_abort) {
      // leave no product in flight (bounded waits; a phase that already completed
      // returns at once)
      if (last1 >= 0) mbar_wait(bar1, (uint32_t)(last1 & 1));
      if (last32 >= 0) { mbar_wait(bar3, (uint32_t)(last32 & 1)); mbar_wait(bar2, (uint32_t)(last32 & 1)); }
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp < 8 && *s_abort == 0) {
    float* dst = a.S_final + (((int64_t)n * H + h) * DKT + i) * DV + col0 + jc;
#pragma unroll
    for (int j = 0; j < NC; j += 4) *reinterpret_cast<float4*>(dst + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
  }
  if (warp == PRODUCER) tmem_dealloc(tmem, 256);
}

// SM count of the current device, looked up once per device.
cudaError_t device_sms(int* sms) {
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

// [T][cols] bf16 tensor map with a box of box_x columns x 64 rows
bool make_map(CUtensorMap* m, const void* base, int64_t T, int64_t cols, int box_x, bool swizzle128) {
  return make_map_2d(m, base, T, cols, 2, box_x, 64, swizzle128);
}

template <int DV>
cudaError_t launch_prep_dv(const PrefillArgs& a, const PrefillSched& sched, unsigned char* ws, int total_chunks,
                           cudaStream_t s) {
  if (total_chunks <= 0) return cudaSuccess;
  PrepMaps maps;
  if (!make_map(&maps.k, a.k, a.T, (int64_t)a.H * DKT, 64, true) ||
      !make_map(&maps.q, a.q, a.T, (int64_t)a.H * DKT, 64, true) ||
      !make_map(&maps.g, a.g, a.T, (int64_t)a.H * DKT, DKT, false) ||
      !make_map(&maps.v, a.v, a.T, (int64_t)a.H * DV, 64, true))
    return cudaErrorInvalidValue;
  auto prep = a.mode == KDA_MODE_DECAY_FIRST ? kda_chunk_prep_kernel<DV, true> : kda_chunk_prep_kernel<DV, false>;
  cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.H * total_chunks;
  if (items > INT32_MAX) return cudaErrorInvalidValue;
  prep<<<(unsigned)items, PNT, P_SMEM, s>>>(a, sched, ws, maps);
  return cudaGetLastError();
}

template <int DV, int DVS>
cudaError_t launch_chain_cols(const PrefillArgs& a, const PrefillSched& sched, const unsigned char* ws,
                              cudaStream_t s) {
  auto chain = kda_chain_kernel<DV, DVS>;
  cudaError_t e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the chain's CTAs may be scheduled while the
  // preceding kernel's last CTAs run; each waits (griddepcontrol.wait) before it
  // reads any memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(DV / DVS, a.H, sched.n_seqs);
  cfg.blockDim = dim3(CNT);
  cfg.dynamicSmemBytes = C_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, chain, a, sched, ws);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DV>
cudaError_t launch_chain_dv(const PrefillArgs& a, const PrefillSched& sched, const unsigned char* ws, cudaStream_t s) {
  int cols = prefill_chain_columns();
  if (cols == 0) {
    // one CTA per SM at most: 32-column slices while twice the 64-column grid still fits
    int sms = 0;
    cudaError_t e = device_sms(&sms);
    if (e != cudaSuccess) return e;
    cols = 2 * (int64_t)(DV / 64) * a.H * sched.n_seqs <= sms ? 32 : 64;
  }
  return cols == 32 ? launch_chain_cols<DV, 32>(a, sched, ws, s) : launch_chain_cols<DV, 64>(a, sched, ws, s);
}

template <int DV>
cudaError_t launch_dv(const PrefillArgs& a, const PrefillSched& sched, unsigned char* ws, int total_chunks,
                      cudaStream_t s) {
  cudaError_t e = launch_prep_dv<DV>(a, sched, ws, total_chunks, s);
  if (e != cudaSuccess) return e;
  return launch_chain_dv<DV>(a, sched, ws, s);
}

}  // namespace

bool prefill_tc_supported(int dk, int dv, int dtype) {
  return dtype == KDA_BF16 && dk == 128 && (dv == 64 || dv == 128);
}

int64_t prefill_tc_image_bytes(int dv) { return img_bytes(dv); }

cudaError_t launch_prefill_tc(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s, bool* handled) {
  *handled = prefill_tc_supported(a.dk, a.dv, a.dtype) && a.workspace != nullptr;
  if (!*handled) return cudaSuccess;
  if (sched.n_seqs == 0 || a.H == 0) return cudaSuccess;
  const int total_chunks = sched.chunk_base[sched.n_seqs];
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  return a.dv == 128 ? launch_dv<128>(a, sched, ws, total_chunks, s)
                     : launch_dv<64>(a, sched, ws, total_chunks, s);
}

cudaError_t launch_prefill_tc_prep(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s) {
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  const int total = sched.chunk_base[sched.n_seqs];
  return a.dv == 128 ? launch_prep_dv<128>(a, sched, ws, total, s) : launch_prep_dv<64>(a, sched, ws, total, s);
}

cudaError_t launch_prefill_tc_chain(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s) {
  if (sched.n_seqs == 0 || a.H == 0) return cudaSuccess;
  const unsigned char* ws = static_cast<const unsigned char*>(a.workspace);
  return a.dv == 128 ? launch_chain_dv<128>(a, sched, ws, s) : launch_chain_dv<64>(a, sched, ws, s);
}

int read_and_clear_device_errors(int* flags) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flags, tc::g_kda_device_error, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  e = cudaMemcpyToSymbol(tc::g_kda_device_error, &zero, sizeof(int));
  return (int)e;
}

}  // namespace kda

// ---------------------------------------------------------------------------
// Fixed device scratch for kda_prefill_chunked_noalloc: callers that cannot
// allocate device memory at call time get the chunk images from this array.
// Device code could name it directly; host code needs its device address,
// which is looked up once per device (with that device current) and kept.
// ---------------------------------------------------------------------------
namespace kda {
namespace {
constexpr unsigned long long kNoallocBytes = KDA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on error).
void* noalloc_scratch(int* cuda_err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *cuda_err = e != cudaSuccess ? (int)e : (int)cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *cuda_err = e != cudaSuccess ? (int)e : (int)cudaErrorInvalidSymbol;
      return nullptr;
    }
    g_noalloc_ptr[dev] = p;
  }
  *cuda_err = 0;
  return g_noalloc_ptr[dev];
}
}  // namespace
}  // namespace kda

extern "C" int kda_prefill_chunked_noalloc(const float* S0, const void* q, const void* k, const void* v,
                                           const void* g, const void* beta, const int32_t* cu_seqlens,
                                           int n_seqs, int64_t T, int H, int dk, int dv, int dtype,
                                           int chunk, int ckpt_stride, void* o, float* S_final,
                                           void* page_pool, int64_t page_bytes,
                                           const int32_t* ckpt_page_ids, int32_t* ckpt_pos,
                                           int64_t num_ckpt, int mode, kda_stream_t stream) {
  // the same argument checks (and errors) as kda_prefill_chunked come first
  if (int st = kda::validate_prefill(S0, q, k, v, g, beta, cu_seqlens, n_seqs, T, H, dk, dv, dtype, chunk,
                                     ckpt_stride, o, S_final, page_pool, page_bytes, ckpt_page_ids, num_ckpt, mode))
    return st;
  const int64_t need = kda_prefill_workspace_bytes(cu_seqlens, n_seqs, T, H, dk, dv, dtype);
  if (need < 0) return (int)need;
  void* ws = nullptr;
  if (need > 0) {
    if ((unsigned long long)need > kda::kNoallocBytes) {
      char msg[256];
      snprintf(msg, sizeof(msg),
               "kda_prefill_chunked_noalloc: this call needs %lld bytes of scratch but the built-in "
               "scratch holds %llu bytes; split the batch or use kda_prefill_chunked with a workspace",
               (long long)need, kda::kNoallocBytes);
      return kda::set_error(KDA_ERR_SHAPE, msg);
    }
    int cerr = 0;
    ws = kda::noalloc_scratch(&cerr);
    if (ws == nullptr) {
      char msg[256];
      snprintf(msg, sizeof(msg), "kda_prefill_chunked_noalloc: scratch address lookup failed: %s",
               cudaGetErrorString((cudaError_t)cerr));
      return kda::set_error(KDA_ERR_CUDA, msg);
    }
  }
  return kda_prefill_chunked(S0, q, k, v, g, beta, cu_seqlens, n_seqs, T, H, dk, dv, dtype, chunk,
                             ckpt_stride, o, S_final, page_pool, page_bytes, ckpt_page_ids, ckpt_pos,
                             num_ckpt, ws, ws ? (int64_t)kda::kNoallocBytes : 0, mode, stream);
}
