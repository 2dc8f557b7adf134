// Sequence-parallel prefill of one long sequence on one GPU (the context-parallel
// prefix scan of "Kimi Linear 的 KDA 缓存", section "预填充为什么能分块并行": every
// token transition is a diagonal matrix minus a rank-one matrix, so the state after
// a segment is affine in the state before it, S_end = M S_start + L; the
// serve-module demo page's KCP passes one (H, dk, dv) state per rank whatever the
// length).
//
// The sequence is cut into P segments of whole chunks (whole checkpoint strides).
//   1. The chunk images of every chunk (chunk-parallel prep), once.
//   2. One chain launch over pseudo-sequences: segment 0 for real from S0 (outputs,
//      checkpoints, its final state = the start of segment 1); for each segment
//      1 .. P-2 its local state L_j (zero start) and its transition M_j, run as
//      dk / dv pseudo-sequences with the beta U term dropped, each starting from a
//      block of dv columns of the identity (their final states are M_j's columns).
//   3. The scan X_{j+1} = M_j X_j + L_j on the tensor cores (tf32 products with X
//      split into a tf32 part and its fp32 remainder, fp32 accumulation; one CTA per
//      head and 32 columns).
//   4. One chain launch over segments 1 .. P-1 from their starts X_j: outputs,
//      checkpoints, and the last segment's final state.
// Steps 2 and 4 each run a 1/P-long chain per (pseudo-)sequence in parallel, so a
// sequence whose heads occupy few SMs finishes in about 2/P of the serial chain's
// time; the prep is shared.
#include "kda_internal.h"
#include "kda_tc.cuh"
#include "kda_tmap.h"
#include "../../include/kda.h"

#include <algorithm>

namespace kda {
namespace {

struct ScanPlan {
  int64_t nch;      // 64-token chunks of the sequence
  int seg;          // chunks per segment
  int P;            // segments
  int nb;           // dk / dv: pseudo-sequences per transition
  int nA;           // pseudo-sequences of the first chain launch
};

ScanPlan make_plan(int64_t len, int dk, int dv, int ckpt_stride, int segments) {
  ScanPlan p{};
  p.nch = (len + 63) / 64;
  const int G = ckpt_stride > 0 ? ckpt_stride / 64 : 1;
  const int64_t want = std::max(1, segments);
  int64_t seg = (p.nch + want - 1) / want;
  seg = (seg + G - 1) / G * G;
  p.seg = (int)std::max<int64_t>(seg, 1);
  p.P = (int)((p.nch + p.seg - 1) / p.seg);
  p.nb = dk / dv;
  p.nA = p.P >= 3 ? 1 + (p.P - 2) * (1 + p.nb) : 0;
  return p;
}

int64_t up256(int64_t x) { return (x + 255) / 256 * 256; }

// start states of the first chain launch: S0 for segment 0, zeros for the local
// states, identity column blocks for the transitions
__global__ void scan_init_kernel(const float* __restrict__ S0, float* __restrict__ S0A, int H, int dk, int dv,
                                 int nA, int nb) {
  const int64_t HS = (int64_t)H * dk * dv;
  const int64_t total = (int64_t)nA * HS;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int slot = (int)(e / HS);
    const int64_t r = e - slot * HS;                       // (h dk + i) dv + c
    const int c = (int)(r % dv), i = (int)((r / dv) % dk);
    float v = 0.f;
    if (slot == 0) {
      v = S0 != nullptr ? S0[r] : 0.f;
    } else {
      const int q = (slot - 1) % (1 + nb);
      if (q > 0) v = (i == (q - 1) * dv + c) ? 1.f : 0.f;
    }
    S0A[e] = v;
  }
}

// X_1 = segment 0's final state; X_{j+1} = M_j X_j + L_j for j = 1 .. P-2, on the
// tensor cores.  One CTA of 128 threads per (head, 32 state columns); thread i owns
// row i.  M_j (fp32, DK x DK) is brought by TMA as the K-major A operand of a
// kind::tf32 product (boxes of 32 columns x 128 rows, 128-byte swizzle), one step
// ahead into a two-stage buffer.  X_j is the MN-major B operand (32 columns of
// 128 bytes per K row) in two parts, X_hi = X rounded to tf32 and X_lo = X - X_hi,
// side by side as one N = 64 operand (two 128-byte atoms), so one product gives
// M_j X_hi and M_j X_lo in TMEM columns 0-31 and 32-63 and their sum keeps X at
// fp32 precision (M_j enters at tf32, relative 2^-11); the readback adds L_j.
constexpr int SCAN_NT = 128;
constexpr uint32_t SC_M = 0;                    // 2 x 64 KB: M_j, M_{j+1}
constexpr uint32_t SC_XH = 131072;              // 16 KB: X_hi, MN-major (mn = 32 columns, K = 128 rows)
constexpr uint32_t SC_XL = SC_XH + 16384;       // 16 KB: X_lo, the operand's second MN atom
constexpr uint32_t SC_MISC = SC_XL + 16384;     // mbarriers, TMEM slot
constexpr uint32_t SC_SMEM = SC_MISC + 64 + 1024;

// tf32 x tf32 -> fp32, A K-major, B MN-major
__host__ __device__ constexpr uint32_t scan_idesc(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (1u << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_tf32_w(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; .reg .b32 r; elect.sync r|e, 0xffffffff; setp.ne.b32 p, %4, 0; "
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p; }"
      :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ float tf32_round(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}
// byte offset of (K row k, column c) in an MN-major 4-byte tile of 32 columns
__device__ __forceinline__ uint32_t off_x(int k, int c) {
  return (uint32_t)((k >> 3) * 1024 + (k & 7) * 128 + ((((c >> 2) ^ (k & 7))) << 4) + (c & 3) * 4);
}

template <int DK>
__global__ void __launch_bounds__(SCAN_NT, 1) scan_kernel(const __grid_constant__ CUtensorMap mmap,
                                                          const float* __restrict__ SfA, float* __restrict__ XC,
                                                          int H, int dv, int P, int nb) {
  static_assert(DK == SCAN_NT, "one thread per state row");
  using namespace tc;
  extern __shared__ unsigned char scan_smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)scan_smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t mbar_m = smem_u32(sm + SC_MISC);          // two M stages landed
  const uint32_t mbar_d = smem_u32(sm + SC_MISC + 16);     // product done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SC_MISC + 32);
  const int h = blockIdx.x, c0 = blockIdx.y * 32, i = threadIdx.x, warp = i >> 5;
  const int64_t HS = (int64_t)H * DK * dv;
  constexpr uint32_t ID = scan_idesc(128, 64);

  // the M_j boxes: K block kb (columns 32 kb ..) is column block b = 32 kb / dv of
  // the transition's pseudo-sequences, at column 32 kb % dv
  auto load_m = [&](int j, int st) {
    const int64_t ls = 1 + (int64_t)(j - 1) * (1 + nb);
    const uint32_t mb = mbar_m + 8 * st;
    mbar_expect_tx(mb, DK * DK * 4);
#pragma unroll
    for (int kb = 0; kb < DK / 32; ++kb) {
      const int b = 32 * kb / dv, x = 32 * kb % dv;
      tma_load_2d(smem_u32(sm + SC_M + st * 65536 + kb * 16384), &mmap, x, (int)((ls + 1 + b) * H + h) * DK, mb);
    }
  };
  auto put_x = [&](const float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = tf32_round(x[4 * q + e]);
        lo[e] = x[4 * q + e] - hi[e];
      }
      *reinterpret_cast<float4*>(sm + SC_XH + off_x(i, 4 * q)) = make_float4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<float4*>(sm + SC_XL + off_x(i, 4 * q)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
    }
  };

  if (i == 0) {
    mbar_init(mbar_m, 1);
    mbar_init(mbar_m + 8, 1);
    mbar_init(mbar_d, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(smem_u32(tslot), 64);
  float x[32];
  {
    const int64_t off = ((int64_t)h * DK + i) * dv + c0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(SfA + off + 4 * q);
      x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
      *reinterpret_cast<float4*>(XC + off + 4 * q) = v;
    }
  }
  put_x(x);
  fence_async_smem();
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;
  int issued = 0;                                          // M loads issued (thread 0)
  if (i == 0 && P >= 3) { load_m(1, 0); issued = 1; }
  bool ok = true;
  for (int j = 1; j <= P - 2 && ok; ++j) {
    const int st = (j - 1) & 1;
    const int64_t ls = 1 + (int64_t)(j - 1) * (1 + nb);
    float l[32];
    const int64_t lo_off = ls * HS + ((int64_t)h * DK + i) * dv + c0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(SfA + lo_off + 4 * q);
      l[4 * q] = v.x; l[4 * q + 1] = v.y; l[4 * q + 2] = v.z; l[4 * q + 3] = v.w;
    }
    // the next transition into the other stage (its last reader, step j - 1's
    // product, is complete)
    if (i == 0 && j + 1 <= P - 2) { load_m(j + 1, st ^ 1); issued = j + 1; }
    if (warp == 0) {
      const bool landed = __all_sync(0xffffffffu, mbar_wait(mbar_m + 8 * st, (uint32_t)(((j - 1) >> 1) & 1)));
      if (landed) {
        fence_after();
        const uint32_t mb = smem_u32(sm + SC_M + st * 65536);
        const uint32_t xh = smem_u32(sm + SC_XH);
        // B: [X_hi | X_lo], the second 128-byte MN atom LBO = SC_XL - SC_XH bytes on
#pragma unroll
        for (int k = 0; k < DK / 8; ++k)
          mma_tf32_w(tmem, desc_k(mb, 128, k), desc_sw128(xh + 1024 * k, SC_XL - SC_XH, 1024), ID, k > 0);
        mma_commit_w(mbar_d);
      }
      ok = landed;
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok) break;
    ok = __syncthreads_and(mbar_wait(mbar_d, (uint32_t)((j - 1) & 1))) != 0;
    if (!ok) break;
    fence_after();
    float d[32], dl[32];
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16), d);
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32, dl);
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] = (d[e] + dl[e]) + l[e];
    const int64_t off = (int64_t)j * HS + ((int64_t)h * DK + i) * dv + c0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4*>(XC + off + 4 * q) = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    put_x(x);
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
  }
  if (i == 0 && !ok) {
    // leave no copy in flight into this CTA's shared memory: the last load of each
    // stage (bounded waits; a phase already seen returns at once)
    for (int jj = max(1, issued - 1); jj <= issued; ++jj)
      mbar_wait(mbar_m + 8 * ((jj - 1) & 1), (uint32_t)(((jj - 1) >> 1) & 1));
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace

// OR the scan kernel's device error word (its bounded waits) into *flags and clear it.
int read_and_clear_scan_errors(int* flags) {
  int word = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&word, tc::g_kda_device_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(tc::g_kda_device_error, &zero, sizeof(int));
  *flags |= word;
  return (int)e;
}

// The segment count asked of make_plan when the caller leaves it open: the most
// segments whose first chain launch still fits one CTA per SM.
int prefill_scan_segments(int64_t len, int H, int dk, int dv, int ckpt_stride, int n_sm) {
  const int64_t nch = (len + 63) / 64;
  for (int P = (int)std::min<int64_t>(64, nch / 4); P >= 3; --P) {
    const ScanPlan p = make_plan(len, dk, dv, ckpt_stride, P);
    if (p.P < 3 || p.nA > kMaxSeqs) continue;
    if ((int64_t)p.nA * H * (dv / 64) <= n_sm) return P;
  }
  return 1;
}

int64_t prefill_scan_scratch_bytes(int64_t len, int H, int dk, int dv, int ckpt_stride, int segments) {
  const ScanPlan p = make_plan(len, dk, dv, ckpt_stride, segments);
  if (p.P < 3) return 0;
  const int64_t HS = (int64_t)H * dk * dv * 4;
  return 2 * up256(p.nA * HS) + 2 * up256((int64_t)(p.P - 1) * HS);
}

cudaError_t launch_prefill_tc_scan(const PrefillArgs& a, int64_t len, int segments, void* scratch, cudaStream_t s) {
  static thread_local PrefillSched sched;
  const ScanPlan p = make_plan(len, a.dk, a.dv, a.ckpt_stride, segments);
  if (p.nA > kMaxSeqs || p.P - 1 > kMaxSeqs) return cudaErrorInvalidValue;
  // chunk images of the whole sequence
  sched.n_seqs = 1;
  sched.order[0] = 0;
  sched.start[0] = 0;
  sched.len[0] = (int32_t)len;
  sched.ckpt_base[0] = 0;
  sched.chunk_base[0] = 0;
  sched.chunk_base[1] = (int32_t)p.nch;
  sched.flags[0] = kSeqEmit;
  sched.pos_base[0] = 0;
  cudaError_t e = launch_prefill_tc_prep(a, sched, s);
  if (e != cudaSuccess || p.P < 3) return e != cudaSuccess ? e : launch_prefill_tc_chain(a, sched, s);

  const int64_t HS = (int64_t)a.H * a.dk * a.dv;
  char* base = static_cast<char*>(scratch);
  float* S0A = reinterpret_cast<float*>(base);
  float* SfA = reinterpret_cast<float*>(base + up256(p.nA * HS * 4));
  float* XC = reinterpret_cast<float*>(base + 2 * up256(p.nA * HS * 4));
  float* SfC = reinterpret_cast<float*>(base + 2 * up256(p.nA * HS * 4) + up256((int64_t)(p.P - 1) * HS * 4));
  const int seg_tok = p.seg * 64;

  // ---- first chain launch: segment 0 for real, local states and transitions ----
  scan_init_kernel<<<1024, 256, 0, s>>>(a.S0, S0A, a.H, a.dk, a.dv, p.nA, p.nb);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  sched.n_seqs = p.nA;
  for (int n = 0; n < p.nA; ++n) {
    const int j = n == 0 ? 0 : 1 + (n - 1) / (1 + p.nb);   // segment of pseudo-sequence n
    const int q = n == 0 ? 0 : (n - 1) % (1 + p.nb);        // 0: local state, > 0: transition block
    sched.order[n] = n;
    sched.start[n] = j * seg_tok;
    sched.len[n] = seg_tok;
    sched.ckpt_base[n] = 0;
    sched.chunk_base[n] = j * p.seg;
    sched.flags[n] = n == 0 ? kSeqEmit : (q > 0 ? kSeqNoU : (uint8_t)0);
    sched.pos_base[n] = j * seg_tok;
  }
  sched.chunk_base[p.nA] = (int32_t)p.nch;
  PrefillArgs aA = a;
  aA.S0 = S0A;
  aA.S_final = SfA;
  if ((e = launch_prefill_tc_chain(aA, sched, s)) != cudaSuccess) return e;

  // ---- scan of the segment starts ----
  auto kern = scan_kernel<128>;                            // the tensor-core chain has dk = 128
  CUtensorMap mmap;                                        // the transitions' states as [rows][dv] fp32
  if (!make_map_2d(&mmap, SfA, (int64_t)p.nA * a.H * a.dk, a.dv, 4, 32, 128, true)) return cudaErrorInvalidValue;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SC_SMEM)) != cudaSuccess)
    return e;
  kern<<<dim3(a.H, a.dv / 32), SCAN_NT, SC_SMEM, s>>>(mmap, SfA, XC, a.H, a.dv, p.P, p.nb);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  // ---- second chain launch: segments 1 .. P-1 from their starts ----
  sched.n_seqs = p.P - 1;
  for (int n = 0; n < p.P - 1; ++n) {
    const int j = n + 1;
    const int64_t st = (int64_t)j * seg_tok;
    sched.order[n] = n;                                      // equal lengths, the last one shorter
    sched.start[n] = (int32_t)st;
    sched.len[n] = (int32_t)std::min<int64_t>(seg_tok, len - st);
    sched.ckpt_base[n] = a.ckpt_stride > 0 ? (int32_t)(st / a.ckpt_stride) : 0;
    sched.chunk_base[n] = j * p.seg;
    sched.flags[n] = kSeqEmit;
    sched.pos_base[n] = (int32_t)st;
  }
  sched.chunk_base[p.P - 1] = (int32_t)p.nch;
  PrefillArgs aC = a;
  aC.S0 = XC;
  aC.S_final = SfC;
  if ((e = launch_prefill_tc_chain(aC, sched, s)) != cudaSuccess) return e;
  return cudaMemcpyAsync(a.S_final, SfC + (int64_t)(p.P - 2) * HS, HS * 4, cudaMemcpyDeviceToDevice, s);
}

}  // namespace kda
