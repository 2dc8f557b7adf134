// Prefill from host-resident inputs to host-resident outputs, with the copies
// overlapped with the computation.
//
// The token range is cut into segments of at most `segment_tokens` tokens (the
// first one half that, since its copy-in is not overlapped with anything) and
// kHostPieces sequence pieces.  A sequence longer than the room left in a
// segment is cut at a multiple of the checkpoint stride (of the 64-token chunk
// when there are no checkpoints) counted from its own start, so every piece
// chunks and checkpoints exactly as the whole sequence would: the state passed
// from one piece to the next is the fp32 state at the cut, and the results are
// the same bits as one device-resident kda_prefill_chunked call.
//
// Three streams per call: copies in (an internal stream), the prefill of each
// segment (the caller's stream) and copies out (an internal stream), ordered by
// events so that segment i + 1 arrives while segment i is computed and segment
// i - 1 leaves.  Device staging is double-buffered inside the caller's scratch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

constexpr int kHostPieces = 8;            // sequence pieces per segment
constexpr int kMaxDevices = 64;

struct Piece {
  int n;            // sequence
  int32_t a, b;     // tokens [a, b) of the sequence
  int32_t len;      // tokens of the whole sequence
};
struct Segment {
  int64_t t0, t1;   // packed token range
  std::vector<Piece> pieces;
};

int align_of(int ckpt_stride) { return ckpt_stride > 0 ? ckpt_stride : 64; }

int64_t round_segment(int64_t segment_tokens, int ckpt_stride) {
  const int al = align_of(ckpt_stride);
  if (segment_tokens < al) segment_tokens = al;
  return (segment_tokens + al - 1) / al * al;
}

std::vector<Segment> plan(const int32_t* cu, int N, int64_t T, int64_t seg, int ckpt_stride) {
  const int al = align_of(ckpt_stride);
  // the first segment is half as long: its copy-in is the only one nothing hides
  const int64_t first = std::max<int64_t>(al, seg / 2 / al * al);
  std::vector<Segment> out;
  Segment cur{0, 0, {}};
  auto close = [&]() {
    if (!cur.pieces.empty()) out.push_back(cur);
    cur = Segment{cur.t1, cur.t1, {}};
  };
  for (int n = 0; n < N; ++n) {
    const int32_t L = cu ? cu[n + 1] - cu[n] : (int32_t)T;
    int32_t pos = 0;
    do {
      if ((int)cur.pieces.size() == kHostPieces) close();
      const int64_t room = (out.empty() ? first : seg) - (cur.t1 - cur.t0);
      if (L - pos <= room) {
        cur.pieces.push_back({n, pos, L, L});
        cur.t1 += L - pos;
        pos = L;
      } else {
        int64_t cut = (pos + room) / al * al;
        if (cut <= pos) {                   // no aligned cut fits: start a fresh segment
          close();
          continue;
        }
        cur.pieces.push_back({n, pos, (int32_t)cut, L});
        cur.t1 += cut - pos;
        pos = (int32_t)cut;
        close();
      }
    } while (pos < L);
  }
  close();
  return out;
}

struct Layout {                           // byte offsets of one staging parity inside the scratch
  int64_t q, k, g, v, beta, o, S0, Sf, parity_bytes, ws;
};

int64_t up256(int64_t x) { return (x + 255) / 256 * 256; }

Layout layout(int64_t seg, int H, int dk, int dv, int dtype) {
  const int64_t es = dtype == KDA_BF16 ? 2 : 4;
  const int64_t st = (int64_t)kHostPieces * H * dk * dv * 4;
  Layout l{};
  int64_t off = 0;
  l.q = off; off += up256(seg * H * dk * es);
  l.k = off; off += up256(seg * H * dk * es);
  l.g = off; off += up256(seg * H * dk * es);
  l.v = off; off += up256(seg * H * dv * es);
  l.beta = off; off += up256(seg * H * es);
  l.o = off; off += up256(seg * H * dv * es);
  l.S0 = off; off += up256(st);
  l.Sf = off; off += up256(st);
  l.parity_bytes = off;
  l.ws = 2 * off;
  return l;
}

// workspace of the tensor-core path for a segment: at most seg / 64 + kHostPieces chunks
int64_t seg_workspace(int64_t seg, int H, int dk, int dv, int dtype) {
  const int32_t cu[2] = {0, (int32_t)(seg + 64LL * kHostPieces)};
  const int64_t w = kda_prefill_workspace_bytes(cu, 1, cu[1], H, dk, dv, dtype);
  return w < 0 ? w : up256(w);
}

std::mutex g_mu;
cudaStream_t g_copy_in[kMaxDevices] = {}, g_copy_out[kMaxDevices] = {};

int copy_streams(cudaStream_t* in, cudaStream_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return e != cudaSuccess ? (int)e : (int)cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_copy_in[dev]) {
    if ((e = cudaStreamCreateWithFlags(&g_copy_in[dev], cudaStreamNonBlocking)) != cudaSuccess) return (int)e;
    if ((e = cudaStreamCreateWithFlags(&g_copy_out[dev], cudaStreamNonBlocking)) != cudaSuccess) return (int)e;
  }
  *in = g_copy_in[dev];
  *out = g_copy_out[dev];
  return 0;
}

int cuda_fail(cudaError_t e, const char* what) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  return kda::set_error(KDA_ERR_CUDA, msg);
}

}  // namespace

extern "C" int64_t kda_prefill_host_scratch_bytes(int H, int dk, int dv, int dtype, int ckpt_stride,
                                                  int64_t segment_tokens) {
  if (H <= 0 || segment_tokens <= 0 || ckpt_stride < 0 || (ckpt_stride % 64) != 0)
    return kda::set_error(KDA_ERR_ARG, "kda_prefill_host_scratch_bytes: H, segment_tokens > 0 and "
                                       "ckpt_stride a non-negative multiple of 64 required");
  if (!(dk == 32 || dk == 64 || dk == 128) || !(dv == 32 || dv == 64 || dv == 128))
    return kda::set_error(KDA_ERR_SHAPE, "kda_prefill_host_scratch_bytes: dk, dv must be 32, 64 or 128");
  if (dtype != KDA_F32 && dtype != KDA_BF16) return kda::set_error(KDA_ERR_DTYPE, "unsupported dtype");
  const int64_t seg = round_segment(segment_tokens, ckpt_stride);
  const Layout l = layout(seg, H, dk, dv, dtype);
  const int64_t w = seg_workspace(seg, H, dk, dv, dtype);
  if (w < 0) return w;
  return l.ws + w;
}

extern "C" int kda_prefill_chunked_host(const float* S0, const void* q, const void* k, const void* v,
                                        const void* g, const void* beta, const int32_t* cu_seqlens,
                                        int n_seqs, int64_t T, int H, int dk, int dv, int dtype, int chunk,
                                        int ckpt_stride, void* o, float* S_final, void* page_pool,
                                        int64_t page_bytes, const int32_t* ckpt_page_ids, int32_t* ckpt_pos,
                                        int64_t num_ckpt, void* scratch, int64_t scratch_bytes,
                                        int64_t segment_tokens, int mode, kda_stream_t stream) {
  if (chunk != 64) return kda::set_error(KDA_ERR_ARG, "kda_prefill_chunked_host: chunk must be 64");
  const int64_t need_scratch = kda_prefill_host_scratch_bytes(H, dk, dv, dtype, ckpt_stride, segment_tokens);
  if (need_scratch < 0) return (int)need_scratch;
  const int64_t n_ck = kda_num_checkpoints(cu_seqlens, n_seqs, T, ckpt_stride);
  if (n_ck < 0) return (int)n_ck;
  const int N = cu_seqlens ? n_seqs : 1;
  if (N == 0) return KDA_OK;
  if (!S_final || (T > 0 && (!q || !k || !v || !g || !beta || !o)))
    return kda::set_error(KDA_ERR_ARG, "kda_prefill_chunked_host: null input or output pointer");
  if (!scratch || scratch_bytes < need_scratch) {
    char msg[256];
    snprintf(msg, sizeof(msg), "kda_prefill_chunked_host: scratch of %lld bytes needed (have %lld)",
             (long long)need_scratch, (long long)scratch_bytes);
    return kda::set_error(KDA_ERR_SHAPE, msg);
  }
  if (((uintptr_t)scratch & 255) != 0) return kda::set_error(KDA_ERR_ALIGN, "scratch must be 256-byte aligned");
  if (n_ck > 0 && (!page_pool || !ckpt_page_ids || num_ckpt < n_ck))
    return kda::set_error(KDA_ERR_ARG, "kda_prefill_chunked_host: checkpoints need page_pool, ckpt_page_ids and "
                                       "num_ckpt >= the count kda_num_checkpoints gives");

  const int64_t seg = round_segment(segment_tokens, ckpt_stride);
  const Layout lay = layout(seg, H, dk, dv, dtype);
  const int64_t ws_bytes = need_scratch - lay.ws;
  const std::vector<Segment> segs = plan(cu_seqlens, N, T, seg, ckpt_stride);
  const int64_t es = dtype == KDA_BF16 ? 2 : 4;
  const int64_t hs = (int64_t)H * dk * dv;          // floats of one sequence's state
  char* base = static_cast<char*>(scratch);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream), s_in = nullptr, s_out = nullptr;
  if (int e = copy_streams(&s_in, &s_out)) return cuda_fail((cudaError_t)e, "kda_prefill_chunked_host streams");

  const int nseg = (int)segs.size();
  std::vector<cudaEvent_t> ev_in(nseg), ev_comp(nseg), ev_out(nseg);
  int created = 0;
  auto destroy = [&]() {
    for (int i = 0; i < created; ++i) {
      cudaEventDestroy(ev_in[i]);
      cudaEventDestroy(ev_comp[i]);
      cudaEventDestroy(ev_out[i]);
    }
  };
  for (; created < nseg; ++created) {
    cudaError_t e = cudaEventCreateWithFlags(&ev_in[created], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_comp[created], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_out[created], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      destroy();
      return cuda_fail(e, "kda_prefill_chunked_host events");
    }
  }
  // the caller's stream may already hold work that wrote the page pool or scratch
  cudaEvent_t ev_start;
  cudaError_t e = cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventRecord(ev_start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_start, 0);
  cudaEventDestroy(ev_start);

  int status = KDA_OK;
  int64_t ck_done = 0;                               // checkpoints emitted before this segment
  std::vector<int32_t> cu_seg;
  for (int i = 0; i < nseg && status == KDA_OK && e == cudaSuccess; ++i) {
    const Segment& sg = segs[i];
    const int p = i & 1;
    char* pb = base + p * lay.parity_bytes;
    const int64_t nt = sg.t1 - sg.t0;
    const int np = (int)sg.pieces.size();
    // ---- in: this segment's projections and the starting states of new sequences ----
    if (i >= 2) e = cudaStreamWaitEvent(s_in, ev_comp[i - 2], 0);
    auto h2d = [&](int64_t off, const void* src, int64_t bytes) {
      if (e == cudaSuccess && bytes > 0)
        e = cudaMemcpyAsync(pb + off, static_cast<const char*>(src) + sg.t0 * (bytes / (nt > 0 ? nt : 1)), bytes,
                            cudaMemcpyHostToDevice, s_in);
    };
    if (nt > 0) {
      h2d(lay.q, q, nt * H * dk * es);
      h2d(lay.k, k, nt * H * dk * es);
      h2d(lay.g, g, nt * H * dk * es);
      h2d(lay.v, v, nt * H * dv * es);
      h2d(lay.beta, beta, nt * H * es);
    }
    for (int j = 0; j < np && e == cudaSuccess; ++j) {
      const Piece& pc = sg.pieces[j];
      if (pc.a == 0 && S0)
        e = cudaMemcpyAsync(pb + lay.S0 + j * hs * 4, S0 + pc.n * hs, hs * 4, cudaMemcpyHostToDevice, s_in);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev_in[i], s_in);
    // ---- compute: states carried from the previous segment, then the prefill ----
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_in[i], 0);
    if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(s, ev_out[i - 2], 0);
    for (int j = 0; j < np && e == cudaSuccess; ++j) {
      const Piece& pc = sg.pieces[j];
      float* dst = reinterpret_cast<float*>(pb + lay.S0) + j * hs;
      if (pc.a > 0) {                                // continues the last piece of the previous segment
        const char* prev = base + (p ^ 1) * lay.parity_bytes;
        const int jl = (int)segs[i - 1].pieces.size() - 1;
        e = cudaMemcpyAsync(dst, prev + lay.Sf + jl * hs * 4, hs * 4, cudaMemcpyDeviceToDevice, s);
      } else if (!S0) {
        e = cudaMemsetAsync(dst, 0, hs * 4, s);
      }
    }
    if (e != cudaSuccess) break;
    cu_seg.assign(1, 0);
    for (const Piece& pc : sg.pieces) cu_seg.push_back(cu_seg.back() + (pc.b - pc.a));
    int64_t ck_seg = 0;
    if (ckpt_stride > 0)
      for (const Piece& pc : sg.pieces) ck_seg += (pc.b - pc.a) / ckpt_stride;
    status = kda_prefill_chunked(reinterpret_cast<const float*>(pb + lay.S0), pb + lay.q, pb + lay.k, pb + lay.v,
                                 pb + lay.g, pb + lay.beta, cu_seg.data(), np, nt, H, dk, dv, dtype, 64,
                                 ckpt_stride, pb + lay.o, reinterpret_cast<float*>(pb + lay.Sf),
                                 ck_seg > 0 ? page_pool : nullptr, page_bytes,
                                 ck_seg > 0 ? ckpt_page_ids + ck_done : nullptr, nullptr, ck_seg,
                                 ws_bytes > 0 ? base + lay.ws : nullptr, ws_bytes, mode, stream);
    ck_done += ck_seg;
    if (status != KDA_OK) break;
    e = cudaEventRecord(ev_comp[i], s);
    // ---- out: outputs and the final states of sequences that end here ----
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_comp[i], 0);
    if (e == cudaSuccess && nt > 0)
      e = cudaMemcpyAsync(static_cast<char*>(o) + sg.t0 * H * dv * es, pb + lay.o, nt * H * dv * es,
                          cudaMemcpyDeviceToHost, s_out);
    for (int j = 0; j < np && e == cudaSuccess; ++j) {
      const Piece& pc = sg.pieces[j];
      if (pc.b == pc.len)
        e = cudaMemcpyAsync(S_final + pc.n * hs, pb + lay.Sf + j * hs * 4, hs * 4, cudaMemcpyDeviceToHost, s_out);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev_out[i], s_out);
  }
  if (status == KDA_OK && e == cudaSuccess && nseg > 0) e = cudaStreamWaitEvent(s, ev_out[nseg - 1], 0);
  if (status == KDA_OK && e == cudaSuccess && ckpt_pos && n_ck > 0) {
    // positions counted from each sequence's start (the segments count from their pieces)
    std::vector<int32_t> pos;
    pos.reserve((size_t)n_ck);
    for (int n = 0; n < N; ++n) {
      const int32_t L = cu_seqlens ? cu_seqlens[n + 1] - cu_seqlens[n] : (int32_t)T;
      for (int32_t t = ckpt_stride; t <= L; t += ckpt_stride) pos.push_back(t);
    }
    // pageable source: staged by the runtime before the call returns, so the
    // vector may go away with this frame
    e = cudaMemcpyAsync(ckpt_pos, pos.data(), pos.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s);
  }
  destroy();
  if (status != KDA_OK) return status;
  if (e != cudaSuccess) return cuda_fail(e, "kda_prefill_chunked_host");
  return KDA_OK;
}
