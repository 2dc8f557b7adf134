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
//   3. The scan X_{j+1} = M_j X_j + L_j in fp32 (one CTA per head and 32 columns).
//   4. One chain launch over segments 1 .. P-1 from their starts X_j: outputs,
//      checkpoints, and the last segment's final state.
// Steps 2 and 4 each run a 1/P-long chain per (pseudo-)sequence in parallel, so a
// sequence whose heads occupy few SMs finishes in about 2/P of the serial chain's
// time; the prep is shared.
#include "kda_internal.h"
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

// X_1 = segment 0's final state; X_{j+1} = M_j X_j + L_j for j = 1 .. P-2.
// One CTA of 256 threads per (head, 32 state columns); X block [DK][32] and M_j
// transposed, [k][i], in shared memory; each thread a 4 x 4 block (rows 4 ti ..,
// columns 4 tc ..): per k one 16-byte read of X's row k and one of M_j's column k
// feed 16 FMAs.
constexpr int SCAN_NT = 256;
template <int DK>
__global__ void __launch_bounds__(SCAN_NT) scan_kernel(const float* __restrict__ SfA, float* __restrict__ XC, int H,
                                                       int dv, int P, int nb) {
  static_assert(DK / 4 * 8 == SCAN_NT, "one thread per 4 x 4 block of a DK x 32 tile");
  extern __shared__ float4 scan_smem4[];
  float* Xs = reinterpret_cast<float*>(scan_smem4);        // [DK][32]
  float* MT = Xs + DK * 32;                                // [DK (k)][DK (i)]
  const int h = blockIdx.x, c0 = blockIdx.y * 32, tid = threadIdx.x;
  const int tc = tid & 7, ti = tid >> 3;                   // column group, row group
  const int64_t HS = (int64_t)H * DK * dv;
  for (int e = tid; e < DK * 32; e += SCAN_NT) {
    const int i = e >> 5, cc = e & 31;
    const int64_t off = ((int64_t)h * DK + i) * dv + c0 + cc;
    const float x = SfA[off];
    Xs[e] = x;
    XC[off] = x;
  }
  __syncthreads();
  // M_j as float4s along k (row i, columns k .. k + 3), consecutive threads on
  // consecutive rows so that the transposed stores hit distinct banks; the loads of
  // M_{j+1} are in flight while step j computes
  constexpr int NM = DK * DK / 4 / SCAN_NT;
  float4 mv[NM];
  auto load_m = [&](int j) {
    const int64_t ls = 1 + (int64_t)(j - 1) * (1 + nb);
#pragma unroll
    for (int u = 0; u < NM; ++u) {
      const int e = tid + SCAN_NT * u, i = e % DK, k = 4 * (e / DK), b = k / dv;
      mv[u] = *reinterpret_cast<const float4*>(SfA + (ls + 1 + b) * HS + ((int64_t)h * DK + i) * dv + (k - b * dv));
    }
  };
  if (P >= 3) load_m(1);
  for (int j = 1; j <= P - 2; ++j) {
    const int64_t ls = 1 + (int64_t)(j - 1) * (1 + nb);    // slot of L_j; M_j's column blocks follow
#pragma unroll
    for (int u = 0; u < NM; ++u) {
      const int e = tid + SCAN_NT * u, i = e % DK, k = 4 * (e / DK);
      MT[(k + 0) * DK + i] = mv[u].x;
      MT[(k + 1) * DK + i] = mv[u].y;
      MT[(k + 2) * DK + i] = mv[u].z;
      MT[(k + 3) * DK + i] = mv[u].w;
    }
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float4 l4 = *reinterpret_cast<const float4*>(SfA + ls * HS + ((int64_t)h * DK + 4 * ti + r) * dv + c0 +
                                                         4 * tc);
      acc[r][0] = l4.x; acc[r][1] = l4.y; acc[r][2] = l4.z; acc[r][3] = l4.w;
    }
    __syncthreads();
    if (j + 1 <= P - 2) load_m(j + 1);
#pragma unroll 8
    for (int k = 0; k < DK; ++k) {
      const float4 x4 = *reinterpret_cast<const float4*>(Xs + k * 32 + 4 * tc);
      const float4 m4 = *reinterpret_cast<const float4*>(MT + k * DK + 4 * ti);
      const float mr[4] = {m4.x, m4.y, m4.z, m4.w}, xc[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(mr[r], xc[q], acc[r][q]);
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float4 o4 = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      *reinterpret_cast<float4*>(Xs + (4 * ti + r) * 32 + 4 * tc) = o4;
      *reinterpret_cast<float4*>(XC + (int64_t)j * HS + ((int64_t)h * DK + 4 * ti + r) * dv + c0 + 4 * tc) = o4;
    }
    __syncthreads();
  }
}

}  // namespace

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
  const int smem = (a.dk * 32 + a.dk * a.dk) * 4;
  if (smem > 48 * 1024 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  kern<<<dim3(a.H, a.dv / 32), SCAN_NT, smem, s>>>(SfA, XC, a.H, a.dv, p.P, p.nb);
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
