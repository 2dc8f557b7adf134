"""Seeded synthetic inputs for the KDA gated delta rule.

This module draws random numbers and nothing else: it holds none of the
recurrence's arithmetic, so that both the fp64 oracle and the CUDA path can be
fed from it without sharing any of the method.

Value distributions follow the workloads of the KDA serve-module demo page
("【轻量化复刻大模型 / KIMI K3】Serve 模块交互式演示", §1.3: alpha = g_min *
sigmoid(.) in [g_min, 0], beta = sigmoid(.) in [0, 1]) and of the Kimi Linear
cache page ("Kimi Linear 的 KDA 缓存", section "KDA 的递推与充分状态": Q and K
arrive L2-normalised, one gate per key channel):

* q, k ~ N(0, 1), then L2-normalised over the key dimension per (token, head);
* v ~ N(0, 1);
* g = g_min * sigmoid(N(0, 1)) per key channel, g_min = -5;
* beta = sigmoid(N(0, 1));
* states ~ N(0, std) in fp32 (std 0.1 or 0.05 by workload, 0 for a cold start).

Arrays are produced by torch generators (seeded, deterministic on one device
type) in float64, then rounded once to the requested storage dtype.  The oracle
consumes exactly those rounded values upcast to float64, the GPU path the
rounded values themselves.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

G_MIN = -5.0


def _gen(seed: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return gen


def _normal(shape, gen, device, dtype=torch.float64):
    return torch.randn(*shape, generator=gen, device=device, dtype=dtype)


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def _draw_projections(lead, dk, dv, dtype, gen, device, g_min, work_dtype):
    q = _unit_rows(_normal((*lead, dk), gen, device, work_dtype))
    k = _unit_rows(_normal((*lead, dk), gen, device, work_dtype))
    v = _normal((*lead, dv), gen, device, work_dtype)
    g = g_min * torch.sigmoid(_normal((*lead, dk), gen, device, work_dtype))
    beta = torch.sigmoid(_normal(tuple(lead), gen, device, work_dtype))
    return {n: t.to(dtype).contiguous() for n, t in
            dict(q=q, k=k, v=v, g=g, beta=beta).items()}


def _state(shape, std, gen, device, work_dtype):
    if std == 0.0:
        return torch.zeros(*shape, device=device, dtype=torch.float32)
    return (std * _normal(shape, gen, device, work_dtype)).to(torch.float32).contiguous()


def decode_inputs(B, H, dk, dv, dtype=torch.float32, seed=0, device="cpu",
                  state_std=0.05, g_min=G_MIN):
    """One decode step: S (B,H,dk,dv) fp32; q,k,g (B,H,dk); v (B,H,dv); beta (B,H)."""
    work = torch.float64 if torch.device(device).type == "cpu" else torch.float32
    gen = _gen(seed, device)
    S = _state((B, H, dk, dv), state_std, gen, device, work)
    proj = _draw_projections((B, H), dk, dv, dtype, gen, device, g_min, work)
    return S, proj


def decode_step_projections(B, H, dk, dv, dtype=torch.bfloat16, seed=0, device="cpu",
                            g_min=G_MIN):
    """Fresh per-step projections for a run of decode steps (no state)."""
    work = torch.float64 if torch.device(device).type == "cpu" else torch.float32
    return _draw_projections((B, H), dk, dv, dtype, _gen(seed, device), device, g_min, work)


@dataclass
class DraftProjections:
    """Cached raw per-draft-step inputs, layout (draft, B, H, D).

    Mirrors the draft-projection cache of the serve-module page (§1.1 route B
    and Tab 4's window layout): step i of the draft lives at index i of the
    leading axis.
    """
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor

    @property
    def draft(self) -> int:
        return int(self.q.shape[0])

    def to(self, *args, **kwargs) -> "DraftProjections":
        return DraftProjections(*(t.to(*args, **kwargs) for t in
                                  (self.q, self.k, self.v, self.g, self.beta)))


def replay_inputs(B, H, dk, dv, draft, dtype=torch.float32, seed=0, device="cpu",
                  state_std=0.1, g_min=G_MIN, n_accepted=None):
    """Committed state, draft projections and per-sequence accepted counts.

    n_accepted ~ Uniform{0..draft} per sequence unless given.
    """
    work = torch.float64 if torch.device(device).type == "cpu" else torch.float32
    gen = _gen(seed, device)
    S = _state((B, H, dk, dv), state_std, gen, device, work)
    p = _draw_projections((draft, B, H), dk, dv, dtype, gen, device, g_min, work)
    proj = DraftProjections(p["q"], p["k"], p["v"], p["g"], p["beta"])
    if n_accepted is None:
        cpu_gen = _gen(seed + 7919, "cpu")
        n_accepted = torch.randint(0, draft + 1, (B,), generator=cpu_gen, dtype=torch.int32)
    n_accepted = torch.as_tensor(n_accepted, dtype=torch.int32).to(device)
    return S, proj, n_accepted


def varlen_lengths(n_seqs=64, lo=512, hi=32768, multiple=64, seed=0):
    """Sequence lengths log-uniform in [lo, hi], rounded to a multiple (host list)."""
    gen = _gen(seed, "cpu")
    u = torch.rand(n_seqs, generator=gen, dtype=torch.float64)
    raw = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    out = []
    for x in raw.tolist():
        L = int(round(x / multiple)) * multiple
        out.append(min(max(L, lo), hi))
    return out


def cu_seqlens_of(lengths):
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return cu


def prefill_inputs(lengths, H, dk, dv, dtype=torch.bfloat16, seed=0, device="cpu",
                   state_std=0.05, g_min=G_MIN):
    """Token-major prefill inputs for one or more packed sequences.

    Returns (S0 (N,H,dk,dv) fp32, dict of q,k,g (T,H,dk), v (T,H,dv), beta (T,H),
    cu_seqlens host list of N+1 ints).
    """
    if isinstance(lengths, int):
        lengths = [lengths]
    work = torch.float64 if torch.device(device).type == "cpu" else torch.float32
    gen = _gen(seed, device)
    N = len(lengths)
    T = sum(int(L) for L in lengths)
    S0 = _state((N, H, dk, dv), state_std, gen, device, work)
    proj = _draw_projections((T, H), dk, dv, dtype, gen, device, g_min, work)
    return S0, proj, cu_seqlens_of(lengths)


def prologue_inputs(lengths, H, dk, dv, w=4, dtype=torch.bfloat16, seed=0, device="cpu",
                    zero_window=False):
    """Raw inputs of the input prologue (ShortConv, activation, L2Norm, gates from logits).

    mixed (T, H (2 dk + dv)) ~ N(0, 1), rows [q | k | v] of the packed sequences;
    conv weight (H (2 dk + dv), w) ~ N(0, 1/w); per-sequence conv windows
    (N, w - 1, H (2 dk + dv)) ~ N(0, 1) (zeros for fresh sequences); gate logits
    (T, H, dk) and beta logits (T, H) ~ N(0, 1).  Returns (dict, cu_seqlens).
    """
    if isinstance(lengths, int):
        lengths = [lengths]
    work = torch.float64 if torch.device(device).type == "cpu" else torch.float32
    gen = _gen(seed, device)
    N = len(lengths)
    T = sum(int(L) for L in lengths)
    C = H * (2 * dk + dv)
    out = {
        "mixed": _normal((T, C), gen, device, work),
        "weight": _normal((C, w), gen, device, work) / math.sqrt(w),
        "window": _normal((N, w - 1, C), gen, device, work),
        "g_logits": _normal((T, H, dk), gen, device, work),
        "beta_logits": _normal((T, H), gen, device, work),
    }
    if zero_window:
        out["window"].zero_()
    return {n: t.to(dtype).contiguous() for n, t in out.items()}, cu_seqlens_of(lengths)


def to_f64_numpy(t: torch.Tensor):
    """The exact stored values, widened to float64 (for the oracle)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
