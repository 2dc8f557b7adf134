// Chunked prefill of the KDA gated delta rule on CUDA cores, fp32 arithmetic.
//
// This is the full-precision path (fp32 projections, or any dtype when the
// fp32 accuracy of every contraction matters).  It follows the chunked form of
// "Kimi Linear 的 KDA 缓存" (section "预填充为什么能分块并行": each token's
// transition is a diagonal minus a rank-one matrix; 64 of them compress into
// WY/UT form with a small lower-triangular solve) and emits chunk-aligned
// checkpoints (section "SGLang：从一次较长的 extend 调用中提取检查点") straight
// into pages in pack_heads layout (KIMI K3 Serve demo page, §1.5).
//
// Per chunk of C = 64 tokens, with Gamma_r the inclusive per-channel cumsum of
// g inside the chunk and G_r = Gamma_r (decay first) or Gamma_{r-1} (undecayed
// delta):
//   A[r,s] = beta_s <k_r, k_s e^{G_r - Gamma_s}>          s < r
//   P[r,s] = <q_r, k_s e^{Gamma_r - Gamma_s}>              s <= r
//   (I + A) Delta = V - (k e^{G}) S                        forward substitution
//   O = (q e^{Gamma}) S + P (beta Delta)
//   S <- e^{Gamma_C} S + (k e^{Gamma_C - Gamma})^T (beta Delta)
// Pairwise decays e^{x_r - y_s} are split as e^{x_r - ref} e^{ref - y_s} with
// one reference per 16-token column block (Gamma at the block's 8th token), so
// each factor stays below e^{8 |g_min|}: finite in fp32 for g >= -10.
//
// One CTA owns one (sequence, head, 32-column slice of dv) and walks the
// sequence's chunks in order with the state slice in shared memory.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "../../include/kda.h"

namespace kda {

// Device error word of this translation unit (same bits as kda_device_errors):
// bit 1 = a gate outside [-10, 0] (or NaN) was read, beyond the range where the
// factor split below stays finite.
static __device__ int g_simt_error = 0;

int read_and_clear_simt_errors(int* flags) {
  int word = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&word, g_simt_error, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_simt_error, &zero, sizeof(int));
  *flags |= word;
  return (int)e;
}

namespace {

constexpr int C = 64;        // chunk length
constexpr int DVS = 32;      // columns of dv per CTA
constexpr int NT = 256;      // threads per CTA
constexpr int DSTR = DVS + 4;  // row stride of the delta buffer (bank-conflict free solve)

template <int DK>
struct SimtSmem {
  static constexpr int KS = DK + 1;                 // padded row stride of chunk x DK arrays
  float Kr[C * KS];      // k, then k e^{Gamma_C - Gamma}
  float Qr[C * KS];      // q, then q e^{Gamma}
  float Gm[C * KS];      // Gamma (inclusive cumsum of g)
  float X[C * KS];       // k e^{ref - Gamma} (per column block), then k e^{G}
  float A[C * (C + 1)];
  float P[C * (C + 1)];
  float S[DK * DVS];
  float D[C * DSTR];     // V, then V - k e^G S, then Delta, then beta Delta
  float QS[C * DVS];
  float beta[C];
  float eGC[DK];
};

template <int DK, typename T>
__global__ void __launch_bounds__(NT, 1)
kda_prefill_simt_kernel(const PrefillArgs a, const PrefillSched sched) {
  using Sm = SimtSmem<DK>;
  constexpr int KS = Sm::KS;
  extern __shared__ float4 smem4[];
  Sm& sm = *reinterpret_cast<Sm*>(smem4);

  const int tid = threadIdx.x;
  const int slice = blockIdx.x, h = blockIdx.y;
  const int seq = sched.order[blockIdx.z];
  const int64_t start = sched.start[seq];
  const int len = sched.len[seq];
  const int H = a.H, DV = a.dv;
  const int col0 = slice * DVS;
  const T* q = reinterpret_cast<const T*>(a.q);
  const T* k = reinterpret_cast<const T*>(a.k);
  const T* v = reinterpret_cast<const T*>(a.v);
  const T* g = reinterpret_cast<const T*>(a.g);
  const T* bt = reinterpret_cast<const T*>(a.beta);
  T* o = reinterpret_cast<T*>(a.o);
  const bool decay_first = a.mode == KDA_MODE_DECAY_FIRST;

  // state slice
  const int64_t sbase = ((int64_t)seq * H + h) * DK * DV + col0;
  for (int e = tid; e < DK * DVS; e += NT) {
    const int i = e / DVS, j = e % DVS;
    sm.S[e] = a.S0 ? a.S0[sbase + (int64_t)i * DV + j] : 0.f;
  }

  int ck = 0;   // checkpoints emitted so far by this sequence
  bool gate_bad = false;
  for (int c0 = 0; c0 < len; c0 += C) {
    const int L = min(C, len - c0);
    const int64_t t0 = start + c0;
    __syncthreads();
    // ---- 1. load the chunk (tokens past L are zero: no decay, no write) ----
    for (int e = tid; e < C * DK; e += NT) {
      const int r = e / DK, i = e % DK;
      float kv = 0.f, qv = 0.f, gv = 0.f;
      if (r < L) {
        const int64_t off = ((t0 + r) * H + h) * DK + i;
        kv = to_f32(k[off]); qv = to_f32(q[off]); gv = to_f32(g[off]);
        gate_bad |= !(gv >= -10.f && gv <= 0.f);
      }
      sm.Kr[r * KS + i] = kv; sm.Qr[r * KS + i] = qv; sm.Gm[r * KS + i] = gv;
    }
    for (int e = tid; e < C * DVS; e += NT) {
      const int r = e / DVS, j = e % DVS;
      sm.D[r * DSTR + j] = r < L ? to_f32(v[((t0 + r) * H + h) * DV + col0 + j]) : 0.f;
    }
    if (tid < C) sm.beta[tid] = tid < L ? to_f32(bt[(t0 + tid) * H + h]) : 0.f;
    __syncthreads();

    // ---- 2. Gamma = cumsum of g per channel; X = k e^{ref - Gamma} ----
    if (tid < DK) {
      const int i = tid;
      float acc = 0.f;
      for (int r = 0; r < C; ++r) { acc += sm.Gm[r * KS + i]; sm.Gm[r * KS + i] = acc; }
      for (int r = 0; r < C; ++r) {
        const float ref = sm.Gm[((r >> 4) * 16 + 7) * KS + i];
        sm.X[r * KS + i] = sm.Kr[r * KS + i] * expf(ref - sm.Gm[r * KS + i]);
      }
      sm.eGC[i] = expf(sm.Gm[(C - 1) * KS + i]);
    }
    __syncthreads();

    // ---- 3. A and P, one (row, 16-column block) per thread ----
    {
      const int r = tid % C, cb = tid / C;
      float acc_a[16], acc_p[16];
#pragma unroll
      for (int s = 0; s < 16; ++s) { acc_a[s] = 0.f; acc_p[s] = 0.f; }
      if (cb <= (r >> 4)) {
        const int rt = cb * 16 + 7;
        for (int i = 0; i < DK; ++i) {
          const float ref = sm.Gm[rt * KS + i];
          const float Gr = decay_first ? sm.Gm[r * KS + i] : (r ? sm.Gm[(r - 1) * KS + i] : 0.f);
          const float ek = sm.Kr[r * KS + i] * expf(Gr - ref);
          const float eq = sm.Qr[r * KS + i] * expf(sm.Gm[r * KS + i] - ref);
#pragma unroll
          for (int s = 0; s < 16; ++s) {
            const float xs = sm.X[(cb * 16 + s) * KS + i];
            acc_a[s] = fmaf(ek, xs, acc_a[s]);
            acc_p[s] = fmaf(eq, xs, acc_p[s]);
          }
        }
      }
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const int sc = cb * 16 + s;
        sm.A[r * (C + 1) + sc] = sc < r ? sm.beta[sc] * acc_a[s] : 0.f;
        sm.P[r * (C + 1) + sc] = sc <= r ? acc_p[s] : 0.f;
      }
    }
    __syncthreads();

    // ---- 3b. X = k e^{G}, Qr = q e^{Gamma}, Kr = k e^{Gamma_C - Gamma} ----
    for (int e = tid; e < C * DK; e += NT) {
      const int r = e / DK, i = e % DK;
      const float Gam = sm.Gm[r * KS + i];
      const float Gr = decay_first ? Gam : (r ? sm.Gm[(r - 1) * KS + i] : 0.f);
      const float kk = sm.Kr[r * KS + i];
      sm.X[r * KS + i] = kk * expf(Gr);
      sm.Qr[r * KS + i] *= expf(Gam);
      sm.Kr[r * KS + i] = kk * expf(sm.Gm[(C - 1) * KS + i] - Gam);
    }
    __syncthreads();

    // ---- 4. D = V - (k e^G) S,  QS = (q e^Gamma) S ----
    {
      const int j = tid % DVS, rq = tid / DVS;
      float ar[C / 8], aq[C / 8];
#pragma unroll
      for (int m = 0; m < C / 8; ++m) { ar[m] = 0.f; aq[m] = 0.f; }
      for (int i = 0; i < DK; ++i) {
        const float sij = sm.S[i * DVS + j];
#pragma unroll
        for (int m = 0; m < C / 8; ++m) {
          const int r = rq + 8 * m;
          ar[m] = fmaf(sm.X[r * KS + i], sij, ar[m]);
          aq[m] = fmaf(sm.Qr[r * KS + i], sij, aq[m]);
        }
      }
#pragma unroll
      for (int m = 0; m < C / 8; ++m) {
        const int r = rq + 8 * m;
        sm.D[r * DSTR + j] -= ar[m];
        sm.QS[r * DVS + j] = aq[m];
      }
    }
    __syncthreads();

    // ---- 5. forward substitution (I + A) Delta = D, 8 lanes per column ----
    {
      const int j = tid / 8, part = tid % 8;
      for (int r = 1; r < C; ++r) {
        float acc = 0.f;
        for (int s = part; s < r; s += 8) acc = fmaf(sm.A[r * (C + 1) + s], sm.D[s * DSTR + j], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (part == 0) sm.D[r * DSTR + j] -= acc;
        __syncwarp();
      }
    }
    __syncthreads();
    for (int e = tid; e < C * DVS; e += NT) {
      const int r = e / DVS, j = e % DVS;
      sm.D[r * DSTR + j] *= sm.beta[r];
    }
    __syncthreads();

    // ---- 6. outputs and state update ----
    {
      const int j = tid % DVS, rq = tid / DVS;
#pragma unroll
      for (int m = 0; m < C / 8; ++m) {
        const int r = rq + 8 * m;
        float acc = sm.QS[r * DVS + j];
        for (int s = 0; s <= r; ++s) acc = fmaf(sm.P[r * (C + 1) + s], sm.D[s * DSTR + j], acc);
        if (r < L) o[((t0 + r) * H + h) * DV + col0 + j] = from_f32<T>(acc);
      }
      for (int i = rq; i < DK; i += 8) {
        float acc = sm.eGC[i] * sm.S[i * DVS + j];
        for (int s = 0; s < C; ++s) acc = fmaf(sm.Kr[s * KS + i], sm.D[s * DSTR + j], acc);
        sm.S[i * DVS + j] = acc;
      }
    }

    // ---- 7. checkpoint at stride boundaries ----
    const int pos = c0 + L;
    if (a.ckpt_stride > 0 && pos % a.ckpt_stride == 0) {
      __syncthreads();
      const int64_t idx = (int64_t)sched.ckpt_base[seq] + ck;
      ++ck;
      if (idx < a.num_ckpt) {
        float* page = reinterpret_cast<float*>(a.page_pool + (int64_t)a.ckpt_page_ids[idx] * a.page_bytes);
        for (int e = tid; e < DK * DVS; e += NT) {
          const int i = e / DVS, j = e % DVS;
          page[((int64_t)h * DK + i) * DV + col0 + j] = sm.S[e];
        }
        if (h == 0 && slice == 0) {
          const int64_t used = (int64_t)H * DK * DV, total = a.page_bytes / 4;
          for (int64_t e = used + tid; e < total; e += NT) page[e] = 0.f;
          if (tid == 0 && a.ckpt_pos) a.ckpt_pos[idx] = pos;
        }
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < DK * DVS; e += NT) {
    const int i = e / DVS, j = e % DVS;
    a.S_final[sbase + (int64_t)i * DV + j] = sm.S[e];
  }
  if (gate_bad) atomicOr(&g_simt_error, 2);
}

template <int DK, typename T>
cudaError_t launch_simt(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s) {
  auto kern = kda_prefill_simt_kernel<DK, T>;
  const size_t smem = sizeof(SimtSmem<DK>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.dv / DVS, a.H, sched.n_seqs);
  kern<<<grid, NT, smem, s>>>(a, sched);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, const PrefillSched& sched, cudaStream_t s) {
  if (sched.n_seqs == 0 || a.H == 0) return cudaSuccess;
  const bool bf = a.dtype == KDA_BF16;
  switch (a.dk) {
    case 32: return bf ? launch_simt<32, __nv_bfloat16>(a, sched, s) : launch_simt<32, float>(a, sched, s);
    case 64: return bf ? launch_simt<64, __nv_bfloat16>(a, sched, s) : launch_simt<64, float>(a, sched, s);
    case 128: return bf ? launch_simt<128, __nv_bfloat16>(a, sched, s) : launch_simt<128, float>(a, sched, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kda
