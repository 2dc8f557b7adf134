"""fp64 CPU oracle of the KDA gated delta rule.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference leg of ``bench.py`` may import or run this
module.  It shares no code with the CUDA library (``kda_delta_rule_gb300``) and
imports nothing from it; the two meet only in the seeded input generators of
``kda_delta_rule_gb300.inputs``, which hold none of the method's arithmetic.

Every function is the plain definition, written out in float64 NumPy, with no
blocking, fusion or reordering beyond what the cited passage states.

Sources (cited below by these short names):

* [SERVE]  page "【轻量化复刻大模型 / KIMI K3】Serve 模块交互式演示"
  (www.cveoy.top/t/topic/qHUG): §1.1 projection cache vs snapshot and the
  ``snapshot_cost_ratio`` formula; §1.2 ``verify_and_replay``; §1.3 the KDA
  recurrence (``kda_step`` / ``kda_recurrent``); §1.5 the unified page pool,
  ``pack_heads`` / ``unpack_heads``; Tab 3 (§6.4) the three acceptance
  scenarios; Tab 7 ``store_kda`` / ``load_kda`` with a zero-padded tail.
* [CACHE]  page "Kimi Linear 的 KDA 缓存：SGLang、vLLM 与 Mooncake Store 全链路"
  (imreese.github.io/blogs/kimi-kda-cache-sglang-vllm-mooncake-store):
  section "KDA 的递推与充分状态" (decay the old state per key channel first,
  then take the prediction error, then write only the increment; one gate per
  key channel; state [heads, d_k, d_v]); section "预填充为什么能分块并行"
  (each transition is a diagonal minus a rank-one matrix; a chunk's
  transitions compress into WY / UT form with a small lower-triangular solve,
  chunk 64); section "SGLang：从一次较长的 extend 调用中提取检查点"
  (chunk-aligned intermediate states); section "检查点状态池的内存成本"
  (recurrent state kept in FP32).

Modes.  ``mode=0`` (DECAY_FIRST) is [CACHE]'s ordering: S' = Diag(e^g) S,
delta = v - S'^T k, S = S' + beta k delta^T, o = S^T q.  ``mode=1``
(UNDECAYED_DELTA) is [SERVE] §1.3's ordering: delta = v - S_{t-1}^T k,
S = Diag(alpha) S_{t-1} + beta k delta^T, o = S^T q, where alpha is read as the
log-decay g in [g_min, 0] (so the factor is e^g): §1.3 bounds alpha to
[g_min, 0], which only makes sense for a log-decay.

Shapes.  State S: (..., dk, dv), rows = key channels, dv contiguous.
q, k, g: (..., dk); v: (..., dv); beta: (...).
"""
from __future__ import annotations

import numpy as np

DECAY_FIRST = 0
UNDECAYED_DELTA = 1


def _f64(x):
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Token-level recurrence ([SERVE] §1.3, [CACHE] "KDA 的递推与充分状态")
# ---------------------------------------------------------------------------

def kda_step(S, q, k, v, g, beta, mode=DECAY_FIRST):
    """One token of the gated delta rule; returns (o, S_new). S is not modified."""
    S, q, k, v, g, beta = map(_f64, (S, q, k, v, g, beta))
    decay = np.exp(g)[..., :, None]                 # Diag(e^g) on the key rows
    b = beta[..., None, None]
    if mode == DECAY_FIRST:
        S_dec = decay * S
        delta = v - np.einsum("...ij,...i->...j", S_dec, k)
        S_new = S_dec + b * k[..., :, None] * delta[..., None, :]
    elif mode == UNDECAYED_DELTA:
        delta = v - np.einsum("...ij,...i->...j", S, k)
        S_new = decay * S + b * k[..., :, None] * delta[..., None, :]
    else:
        raise ValueError(f"unknown mode {mode}")
    o = np.einsum("...ij,...i->...j", S_new, q)
    return o, S_new


def kda_recurrent(S0, q, k, v, g, beta, mode=DECAY_FIRST, return_states=False):
    """Sequential loop of kda_step over the leading (time) axis of q,k,v,g,beta.

    Returns (o (T, ..., dv), S_T) and, if asked, the states (T+1, ..., dk, dv)
    with states[0] = S0.  [SERVE] §1.2 calls this the standard answer.
    """
    S = _f64(S0).copy()
    T = int(np.shape(q)[0])
    outs, states = [], [S.copy()]
    for t in range(T):
        o, S = kda_step(S, q[t], k[t], v[t], g[t], beta[t], mode)
        outs.append(o)
        if return_states:
            states.append(S.copy())
    dv = np.shape(S)[-1]
    o = np.stack(outs) if outs else np.zeros((0,) + np.shape(S)[:-2] + (dv,))
    if return_states:
        return o, S, np.stack(states)
    return o, S


def kda_decode_step(S, q, k, v, g, beta, mode=DECAY_FIRST):
    """Batched decode: (B,H,...) inputs, one step. Returns (o, S_new)."""
    return kda_step(S, q, k, v, g, beta, mode)


# ---------------------------------------------------------------------------
# Raw-input ring ([SERVE] Tab 4 §7.2: RawInputRing, the streaming window of
# raw draft projections that fold-every-commit replays)
# ---------------------------------------------------------------------------

class RawInputRing:
    """Per-slot window of raw draft projections (q, k, v, g, beta), one entry per step.

    [SERVE] Tab 4 §7.2: during verification each draft step's raw inputs are
    streamed into the window instead of snapshotting the state; once it holds
    ``capacity`` steps a push overwrites the oldest (FIFO), so the size stays
    at ``capacity`` from the capacity-th push on; ``window()`` gives the held
    steps oldest first in the draft-projection layout (draft, B, H, D), which
    is what ``verify_and_replay`` consumes at commit time.
    """

    def __init__(self, capacity):
        if int(capacity) < 1:
            raise ValueError("capacity must be >= 1")
        self.capacity = int(capacity)
        self._steps = []                  # oldest first

    def push(self, q, k, v, g, beta):
        if len(self._steps) == self.capacity:
            self._steps.pop(0)            # full: the oldest step is overwritten
        self._steps.append(tuple(_f64(x).copy() for x in (q, k, v, g, beta)))

    def __len__(self):
        return len(self._steps)

    def reset(self):
        self._steps = []

    def window(self):
        """(q, k, v, g, beta), each stacked to (len, B, H, D) / (len, B, H), oldest first."""
        if not self._steps:
            raise ValueError("empty window")
        return tuple(np.stack([st[i] for st in self._steps]) for i in range(5))


# ---------------------------------------------------------------------------
# Speculative verify and replay ([SERVE] §1.2, Tab 3 §6.4)
# ---------------------------------------------------------------------------

def verify_and_replay(S_committed, q, k, v, g, beta, n, mode=DECAY_FIRST):
    """Clone the committed state and replay the first n draft steps.

    Projections have layout (draft, B, H, D) ([SERVE] §1.1 route B, Tab 4).
    Returns (S_new, out) with out stacked as (B, H, n, dv); n = 0 gives an
    empty output (third axis 0) and S_new equal to S_committed.
    """
    S = _f64(S_committed).copy()          # clone: the committed state is shared
    outs = []
    for i in range(int(n)):
        o, S = kda_step(S, q[i], k[i], v[i], g[i], beta[i], mode)
        outs.append(o)
    lead = np.shape(S)[:-2]
    dv = np.shape(S)[-1]
    if outs:
        out = np.stack(outs, axis=-2)
    else:
        out = np.zeros(lead + (0, dv))
    return S, out


def verify_and_replay_batched(S_committed, q, k, v, g, beta, n_accepted, mode=DECAY_FIRST):
    """Per-sequence accepted counts n_b: one verify_and_replay per sequence b.

    S_committed (B,H,dk,dv); projections (draft,B,H,D); n_accepted (B,).
    Returns S_new (B,H,dk,dv) and out (B,H,draft,dv), zero past n_b.
    """
    S_committed = _f64(S_committed)
    B, H, dk, dv = S_committed.shape
    draft = int(np.shape(q)[0])
    S_new = np.empty_like(S_committed)
    out = np.zeros((B, H, draft, dv))
    for b in range(B):
        n_b = int(min(max(int(n_accepted[b]), 0), draft))
        sl = (slice(None), b)
        S_b, out_b = verify_and_replay(S_committed[b], _f64(q)[sl], _f64(k)[sl], _f64(v)[sl],
                                       _f64(g)[sl], _f64(beta)[sl], n_b, mode)
        S_new[b] = S_b
        out[b, :, :n_b] = out_b
    return S_new, out


# ---------------------------------------------------------------------------
# Explicit transition matrices ([CACHE] "预填充为什么能分块并行": every
# transition is a diagonal matrix minus a rank-one matrix)
# ---------------------------------------------------------------------------

def transition_matrix(k, g, beta, mode=DECAY_FIRST):
    """The dk x dk matrix M_t with S_t = M_t S_{t-1} + beta k v^T (one head)."""
    k, g = _f64(k), _f64(g)
    D = np.diag(np.exp(g))
    kkT = float(beta) * np.outer(k, k)
    if mode == DECAY_FIRST:
        return (np.eye(k.shape[0]) - kkT) @ D
    return D - kkT


def unrolled_products(S0, q, k, v, g, beta, mode=DECAY_FIRST):
    """Brute force for one head: S_t = (M_t...M_1) S0 + sum_s (M_t...M_{s+1}) beta_s k_s v_s^T.

    Builds every product of transition matrices explicitly; o_t = S_t^T q_t.
    Returns (o (T,dv), S_T).  For tiny T only.
    """
    S0 = _f64(S0)
    T = int(np.shape(q)[0])
    dk = S0.shape[0]
    Ms = [transition_matrix(k[t], g[t], beta[t], mode) for t in range(T)]
    outs = []
    S_t = S0
    for t in range(T):
        prod_all = np.eye(dk)
        for m in range(t, -1, -1):
            prod_all = prod_all @ Ms[m]
        S_t = prod_all @ S0
        for s in range(t + 1):
            P = np.eye(dk)
            for m in range(t, s, -1):
                P = P @ Ms[m]
            S_t = S_t + P @ (float(beta[s]) * np.outer(_f64(k[s]), _f64(v[s])))
        outs.append(S_t.T @ _f64(q[t]))
    return np.stack(outs), S_t


def segment_transition(k, g, beta, mode=DECAY_FIRST):
    """Product of the transition matrices of a run of tokens, later tokens on the left:
    the state after the run is segment_transition @ S_before + (the run's state from zero)."""
    k = _f64(k)
    M = np.eye(k.shape[-1])
    for t in range(k.shape[0]):
        M = transition_matrix(k[t], g[t], beta[t], mode) @ M
    return M


def prefill_segment_scan(S0, q, k, v, g, beta, seg_len, mode=DECAY_FIRST):
    """Sequence-parallel form of one head's prefill (context-parallel prefix scan).

    [CACHE] "预填充为什么能分块并行": every token transition is a diagonal matrix minus a
    rank-one matrix, so the state after a segment is affine in the state before it,
    S_end = M S_start + L with M the product of the segment's transitions and L the
    segment's state from zero.  The serve-module page's KCP passes one (H, dk, dv) state
    per rank, independent of length.  Segment starts come from the scan
    X_{j+1} = M_j X_j + L_j, X_0 = S0; each segment's outputs from its own start state.
    Returns (o (T, dv), S_T).
    """
    X = _f64(S0).copy()
    T = int(np.shape(q)[0])
    outs = []
    for a in range(0, T, seg_len):
        b = min(T, a + seg_len)
        o_seg, _ = kda_recurrent(X, q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], mode)
        M = segment_transition(k[a:b], g[a:b], beta[a:b], mode)
        _, L = kda_recurrent(np.zeros_like(X), q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], mode)
        X = M @ X + L
        outs.append(o_seg)
    dv = X.shape[-1]
    return (np.concatenate(outs) if outs else np.zeros((0, dv))), X


# ---------------------------------------------------------------------------
# Chunked WY / UT form ([CACHE] "预填充为什么能分块并行")
# ---------------------------------------------------------------------------

def ut_inverse(A):
    """(I + A)^{-1} for strictly lower-triangular A, by forward substitution.

    This is the small lower-triangular solve of the UT transform: row r of
    T = (I + A)^{-1} is e_r - sum_{s<r} A[r,s] T[s].
    """
    C = A.shape[0]
    T = np.zeros_like(A)
    for r in range(C):
        T[r, r] = 1.0
        for s in range(r):
            T[r] -= A[r, s] * T[s]
    return T


def chunk_step(S, q, k, v, g, beta, mode=DECAY_FIRST):
    """Advance one head's state across one chunk of L tokens in WY / UT form.

    q,k,g (L,dk); v (L,dv); beta (L,). Returns (o (L,dv), S_end).

    With Gamma_r = sum_{s<=r} g_s (per key channel, within the chunk) and
    G_r = Gamma_r (decay-first) or Gamma_{r-1} (undecayed delta; Gamma_{-1}=0),
    the L token steps are equivalent to
      A[r,s] = beta_s <k_r, k_s * e^{G_r - Gamma_s}>     (s < r)
      T      = (I + A)^{-1}                              (UT transform)
      W = T (k * e^{G}),   U = T v                       (WY representation)
      Delta  = U - W S                                   (per-token delta)
      P[r,s] = <q_r, k_s * e^{Gamma_r - Gamma_s}>        (s <= r)
      O      = (q * e^{Gamma}) S + P (beta * Delta)
      S_end  = e^{Gamma_L} * S + (k * e^{Gamma_L - Gamma})^T (beta * Delta)
    Pairwise decays are taken as exp of a difference (never a ratio of exps),
    so no intermediate overflows for any g <= 0.
    """
    S, q, k, v, g, beta = map(_f64, (S, q, k, v, g, beta))
    L = q.shape[0]
    Gam = np.cumsum(g, axis=0)
    G = Gam if mode == DECAY_FIRST else Gam - g
    lower_strict = np.tril(np.ones((L, L), dtype=bool), -1)
    lower = np.tril(np.ones((L, L), dtype=bool), 0)
    # pairwise per-channel decays exp(G_r - Gamma_s) / exp(Gamma_r - Gamma_s), only where s<r / s<=r
    dA = G[:, None, :] - Gam[None, :, :]
    dP = Gam[:, None, :] - Gam[None, :, :]
    EA = np.exp(np.where(lower_strict[:, :, None], dA, -np.inf))   # 0 where s >= r
    EP = np.exp(np.where(lower[:, :, None], dP, -np.inf))          # 0 where s > r
    A = np.einsum("ri,si,rsi->rs", k, k, EA) * beta[None, :]
    P = np.einsum("ri,si,rsi->rs", q, k, EP)
    T = ut_inverse(A)
    W = T @ (k * np.exp(G))
    U = T @ v
    Delta = U - W @ S
    bD = beta[:, None] * Delta
    O = (q * np.exp(Gam)) @ S + P @ bD
    GL = Gam[L - 1]
    S_end = np.exp(GL)[:, None] * S + (k * np.exp(GL[None, :] - Gam)).T @ bD
    return O, S_end


def checkpoint_positions(L, ckpt_stride):
    """Chunk-aligned checkpoint boundaries of one sequence: stride, 2*stride, ... <= L.

    t = 0 is the starting state itself and is not emitted; t = L is emitted when
    L is a multiple of the stride ([CACHE] "SGLang：从一次较长的 extend 调用中提取检查点").
    """
    if ckpt_stride is None or ckpt_stride <= 0:
        return []
    return [ckpt_stride * j for j in range(1, int(L) // int(ckpt_stride) + 1)]


def num_checkpoints(lengths, ckpt_stride):
    return sum(len(checkpoint_positions(L, ckpt_stride)) for L in lengths)


def prefill_chunked(S0, q, k, v, g, beta, cu_seqlens=None, chunk=64, ckpt_stride=512,
                    mode=DECAY_FIRST):
    """Chunked prefill of packed sequences with checkpoint emission.

    S0 (N,H,dk,dv); q,k,g (T,H,dk); v (T,H,dv); beta (T,H); cu_seqlens (N+1,)
    (None: one sequence).  Chunks start at each sequence's first token; the last
    chunk of a sequence may be shorter.  Returns (o (T,H,dv), S_final (N,H,dk,dv),
    ckpts) with ckpts a list of (seq, position, state (H,dk,dv)) in sequence
    order then position order.  Positions count from the sequence's own start.
    """
    S0 = _f64(S0)
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    T, H, _ = q.shape
    if cu_seqlens is None:
        cu_seqlens = [0, T]
    cu = [int(x) for x in cu_seqlens]
    N = len(cu) - 1
    if ckpt_stride and ckpt_stride % chunk:
        raise ValueError("ckpt_stride must be a multiple of chunk")
    o = np.zeros((T, H, v.shape[2]))
    S_final = np.empty_like(S0)
    ckpts = []
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        S = S0[n].copy()                                  # (H,dk,dv); S0 is never written
        pos = 0
        while pos < b - a:
            L = min(chunk, b - a - pos)
            t0 = a + pos
            for h in range(H):
                O, S[h] = chunk_step(S[h], q[t0:t0 + L, h], k[t0:t0 + L, h], v[t0:t0 + L, h],
                                     g[t0:t0 + L, h], beta[t0:t0 + L, h], mode)
                o[t0:t0 + L, h] = O
            pos += L
            if ckpt_stride and pos % ckpt_stride == 0:
                ckpts.append((n, pos, S.copy()))
        S_final[n] = S
    return o, S_final, ckpts


def prefill_recurrent(S0, q, k, v, g, beta, cu_seqlens=None, ckpt_stride=512,
                      mode=DECAY_FIRST):
    """Same contract as prefill_chunked, computed token by token."""
    S0 = _f64(S0)
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    T, H, _ = q.shape
    if cu_seqlens is None:
        cu_seqlens = [0, T]
    cu = [int(x) for x in cu_seqlens]
    o = np.zeros((T, H, v.shape[2]))
    S_final = np.empty_like(S0)
    ckpts = []
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        S = S0[n].copy()
        for t in range(a, b):
            o[t], S = kda_step(S, q[t], k[t], v[t], g[t], beta[t], mode)
            if ckpt_stride and (t + 1 - a) % ckpt_stride == 0:
                ckpts.append((n, t + 1 - a, S.copy()))
        S_final[n] = S
    return o, S_final, ckpts


# ---------------------------------------------------------------------------
# Input prologue: ShortConv, activation, L2Norm, gates from logits.
# [CACHE] "KDA 的递推与充分状态": before the recurrence each layer's input goes
# through a linear projection, a causal short convolution and an activation, and
# Q and K are L2-normalised.  [CACHE] "先统一记号：矩阵状态不等于完整检查点": the
# ShortConv window of a layer at a boundary has kernel size w (the w - 1 most
# recent inputs); "一个逻辑检查点如何展开": SGLang keeps it as
# [layers, slots, kernel_size - 1, qkv_width]; "SGLang：从一次较长的 extend
# 调用中提取检查点": the conv checkpoint is the kernel_size - 1 rows of mixed_qkv
# just before the boundary.  [SERVE] §1.3: alpha = g_min * sigmoid(.) in
# [g_min, 0] (read as the log-decay g), beta = sigmoid(.) in [0, 1].
# Readings where the pages are silent (the equations are stripped): mixed_qkv
# rows are [q (H dk) | k (H dk) | v (H dv)]; the convolution is depthwise over
# time with no bias, y[t, c] = sum_j W[c, j] z[t + j, c] over z = [window; x];
# the activation is none or SiLU; L2Norm is x / sqrt(sum x^2 + eps) over each
# head's dk channels, after the activation.
# ---------------------------------------------------------------------------

ACT_NONE = 0
ACT_SILU = 1


def sigmoid(x):
    x = _f64(x)
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    x = _f64(x)
    return x * sigmoid(x)


def l2norm(x, eps=1e-6):
    """x / sqrt(sum(x^2) + eps) over the last axis."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def short_conv(x, weight, window=None):
    """Causal depthwise convolution of x (T, C) with weight (C, w).

    window (w - 1, C): the inputs just before x (oldest first); None = zeros.
    Returns (y (T, C), window_out (w - 1, C)), window_out being the last w - 1
    rows of [window; x].
    """
    x, weight = _f64(x), _f64(weight)
    T, C = x.shape
    w = weight.shape[1]
    if window is None:
        window = np.zeros((w - 1, C))
    z = np.concatenate([_f64(window), x], axis=0)          # (w - 1 + T, C)
    y = np.zeros((T, C))
    for t in range(T):
        for j in range(w):                                # tap j reads input t - (w - 1) + j
            y[t] += weight[:, j] * z[t + j]
    return y, z[T:].copy()


def gates_from_logits(g_logits, beta_logits, g_min):
    """g = g_min * sigmoid(a) per key channel, beta = sigmoid(b)."""
    return g_min * sigmoid(g_logits), sigmoid(beta_logits)


def input_prep(mixed, weight, window, g_logits, beta_logits, H, dk, dv, g_min,
               act=ACT_SILU, eps=1e-6):
    """One sequence of raw inputs -> the recurrence's (q, k, v, g, beta).

    mixed (T, H (2 dk + dv)) rows [q | k | v]; weight (H (2 dk + dv), w);
    window (w - 1, H (2 dk + dv)) or None; g_logits (T, H, dk); beta_logits (T, H).
    Returns q, k (T, H, dk), v (T, H, dv), g (T, H, dk), beta (T, H) and the
    window after the sequence.
    """
    mixed = _f64(mixed)
    T = mixed.shape[0]
    y, window_out = short_conv(mixed, weight, window)
    if act == ACT_SILU:
        y = silu(y)
    elif act != ACT_NONE:
        raise ValueError(f"unknown activation {act}")
    q = l2norm(y[:, :H * dk].reshape(T, H, dk), eps)
    k = l2norm(y[:, H * dk:2 * H * dk].reshape(T, H, dk), eps)
    v = y[:, 2 * H * dk:].reshape(T, H, dv)
    g, beta = gates_from_logits(g_logits, beta_logits, g_min)
    return q, k, v, g, beta, window_out


def conv_window_at(mixed, window, boundary):
    """The conv checkpoint at `boundary` tokens: the w - 1 rows of [window; mixed]
    that precede it (oldest first)."""
    z = np.concatenate([_f64(window), _f64(mixed)], axis=0)
    wm1 = np.shape(window)[0]
    return z[boundary:boundary + wm1].copy()


# ---------------------------------------------------------------------------
# Page pool packing ([SERVE] §1.5, Tab 6, Tab 7)
# ---------------------------------------------------------------------------

def pack_heads(S):
    """(B,H,dk,dv) -> flat, head-contiguous (row-major over b, h, i, j)."""
    S = np.asarray(S)
    return np.ascontiguousarray(S).reshape(-1).copy()


def unpack_heads(flat, B, H, dk, dv):
    """flat -> (B,H,dk,dv); the exact inverse of pack_heads."""
    n = B * H * dk * dv
    return np.asarray(flat)[:n].reshape(B, H, dk, dv).copy()


def store_kda(state, page_elems):
    """pack_heads into a page of page_elems elements; the tail past the state is zero."""
    flat = pack_heads(state)
    if flat.size > page_elems:
        raise ValueError("state does not fit the page")
    page = np.zeros(page_elems, dtype=flat.dtype)
    page[:flat.size] = flat
    return page


def load_kda(page, B, H, dk, dv):
    return unpack_heads(page, B, H, dk, dv)


# ---------------------------------------------------------------------------
# Byte accounting ([SERVE] §1.1)
# ---------------------------------------------------------------------------

def snapshot_bytes_per_step(H, dk, dv, itemsize):
    """Route A: one full state snapshot per draft step."""
    return H * dk * dv * itemsize


def projection_bytes_per_step(H, dk, dv, itemsize):
    """Route B: the raw (q, k, v, g, beta) of one draft step."""
    return H * (3 * dk + dv + 1) * itemsize


def snapshot_cost_ratio(H, dk, dv):
    """(H dk dv) / (H (3 dk + dv + 1)); independent of draft length and dtype."""
    return (H * dk * dv) / (H * (3 * dk + dv + 1))
