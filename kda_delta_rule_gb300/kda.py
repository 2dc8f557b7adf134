"""Python binding of the KDA C ABI (``include/kda.h``): argument marshalling only.

Every function here checks that its tensors are CUDA tensors of the expected
dtype and layout, allocates missing outputs with PyTorch, and calls the entry
point of the same name in ``libkda.so``.  All computation happens in the
library's kernels; there is no CPU path.  Importing this module raises if the
library has not been built (``python -m kda_delta_rule_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkda.so")

KDA_OK = 0
KDA_F32, KDA_BF16 = 0, 1
DECAY_FIRST, UNDECAYED_DELTA = 0, 1
PAGE_FREE, PAGE_KDA_STATE, PAGE_MLA_KV = 0, 1, 2
LAYOUT_KV, LAYOUT_VK = 0, 1
ACT_NONE, ACT_SILU = 0, 1
MAX_DRAFT = 16
DEVERR_WAIT, DEVERR_GATE = 1, 2


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {message} (status {status})")
        self.status = status


def _load():
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"KDA CUDA library not found at {_LIB_PATH}; build it with "
            "`python -m kda_delta_rule_gb300.build` (needs nvcc for sm_103a)")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, L, D, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float
    sig = {
        "kda_version": ([], I),
        "kda_status_string": ([I], ctypes.c_char_p),
        "kda_last_error": ([], ctypes.c_char_p),
        "kda_decode_step": ([P, P, P, P, P, P, P, I, I, I, I, I, I, P], I),
        "kda_verify_replay": ([P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P], I),
        "kda_verify_replay_layers": ([I, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P], I),
        "kda_decode_step_slots": ([P, L, P, I, P, P, P, P, P, P, I, I, I, I, I, I, P], I),
        "kda_verify_replay_slots": ([I, P, P, L, P, P, I, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P], I),
        "kda_decode_step_fused": ([P, L, P, I, P, P, P, I, P, P, F, I, P, P, P, P, P, P, I, I, I, I, I, I, P], I),
        "kda_prefill_scan": ([P, P, P, P, P, P, L, I, I, I, I, I, I, P, P, P, L, P, P, L, P, L, I, I, P], I),
        "kda_prefill_scan_workspace_bytes": ([L, I, I, I, I, I, I], L),
        "kda_input_prep": ([P, P, I, P, P, P, P, F, I, P, I, L, I, I, I, I, P, P, P, P, P, I, P, L, P], I),
        "kda_num_checkpoints": ([P, I, L, I], L),
        "kda_prefill_chunked": ([P, P, P, P, P, P, P, I, L, I, I, I, I, I, I, P, P, P, L, P, P, L, P, L, I, P], I),
        "kda_prefill_workspace_bytes": ([P, I, L, I, I, I, I], L),
        "kda_prefill_chunked_noalloc": ([P, P, P, P, P, P, P, I, L, I, I, I, I, I, I, P, P, P, L, P, P, L, I, P], I),
        "kda_prefill_host_scratch_bytes": ([I, I, I, I, I, L], L),
        "kda_prefill_chunked_host": ([P, P, P, P, P, P, P, I, L, I, I, I, I, I, I, P, P, P, L, P, P, L, P, L, L, I, P],
                                     I),
        "kda_device_errors": ([ctypes.POINTER(ctypes.c_int)], I),
        "kda_set_prefill_chain_columns": ([I], I),
        "kda_pack_heads": ([P, L, L, P, L, I, I, I, I, P], I),
        "kda_unpack_heads": ([P, P, L, L, I, I, I, I, P], I),
        "kda_pool_create": ([P, L, L, ctypes.POINTER(P)], I),
        "kda_pool_destroy": ([P], I),
        "kda_pool_alloc": ([P, I, L, P], I),
        "kda_pool_free": ([P, L, P], I),
        "kda_pool_num_free": ([P], L),
        "kda_pool_page_kind": ([P, ctypes.c_int32], I),
        "kda_pool_page_ptr": ([P, ctypes.c_int32], P),
        "kda_store_kda": ([P, ctypes.c_int32, P, L, L, I, I, I, I, P], I),
        "kda_load_kda": ([P, ctypes.c_int32, P, L, L, I, I, I, I, P], I),
        "kda_snapshot_cost_ratio": ([I, I, I], D),
        "kda_ring_bytes": ([I, I, I, I, I, I], L),
        "kda_ring_create": ([P, I, I, I, I, I, I, ctypes.POINTER(P)], I),
        "kda_ring_destroy": ([P], I),
        "kda_ring_reset": ([P], I),
        "kda_ring_len": ([P], I),
        "kda_ring_push": ([P, P, P, P, P, P, P], I),
        "kda_ring_window": ([P, P, P, P, P, P, P], I),
        "kda_verify_replay_ring": ([P, P, P, P, P, I, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def _check(status: int, where: str):
    if status != KDA_OK:
        raise KdaError(status, where, _lib.kda_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KDA_F32
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"projections must be float32 or bfloat16, got {t.dtype}")


def _cuda(name, t, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _projections(q, k, v, g, beta, lead):
    dt = q.dtype
    dk = q.shape[-1]
    dv = v.shape[-1]
    _cuda("q", q, dt, (*lead, dk))
    _cuda("k", k, dt, (*lead, dk))
    _cuda("g", g, dt, (*lead, dk))
    _cuda("v", v, dt, (*lead, dv))
    _cuda("beta", beta, dt, tuple(lead))
    return _dtype_code(q), dk, dv


# ---------------------------------------------------------------------------
def kda_decode_step(S, q, k, v, g, beta, o=None, mode=DECAY_FIRST, stream=None):
    """One token for every (b, h) head; S (B,H,dk,dv) fp32 is updated in place. Returns o."""
    B, H, dk, dv = S.shape
    _cuda("S", S, torch.float32)
    code, _, _ = _projections(q, k, v, g, beta, (B, H))
    if o is None:
        o = torch.empty((B, H, dv), device=S.device, dtype=q.dtype)
    _cuda("o", o, q.dtype, (B, H, dv))
    _check(_lib.kda_decode_step(_ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o),
                                B, H, dk, dv, code, mode, _stream(stream, S.device)),
           "kda_decode_step")
    return o


def kda_verify_replay(S_committed, q, k, v, g, beta, n_accepted, S_new=None, out=None,
                      mode=DECAY_FIRST, stream=None):
    """Replay the accepted draft prefix from a clone of S_committed (left untouched).

    Projections (draft,B,H,D); n_accepted int32 (B,). Returns (S_new, out (B,H,draft,dv)).
    """
    B, H, dk, dv = S_committed.shape
    draft = q.shape[0]
    _cuda("S_committed", S_committed, torch.float32)
    code, _, _ = _projections(q, k, v, g, beta, (draft, B, H))
    _cuda("n_accepted", n_accepted, torch.int32, (B,))
    if S_new is None:
        S_new = torch.empty_like(S_committed)
    if out is None:
        out = torch.empty((B, H, draft, dv), device=S_committed.device, dtype=q.dtype)
    _cuda("S_new", S_new, torch.float32, (B, H, dk, dv))
    _cuda("out", out, q.dtype, (B, H, draft, dv))
    _check(_lib.kda_verify_replay(_ptr(S_committed), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _ptr(n_accepted), _ptr(S_new), _ptr(out), draft, B, H, dk, dv,
                                  code, mode, _stream(stream, S_committed.device)),
           "kda_verify_replay")
    return S_new, out


def kda_verify_replay_layers(S_committed, q, k, v, g, beta, n_accepted, S_new=None, out=None,
                             mode=DECAY_FIRST, stream=None):
    """kda_verify_replay for a stack of KDA layers in one launch.

    S_committed (L,B,H,dk,dv) fp32; projections (L,draft,B,H,D); n_accepted int32 (B,) shared
    by the layers. Returns (S_new (L,B,H,dk,dv), out (L,B,H,draft,dv)).
    """
    Lr, B, H, dk, dv = S_committed.shape
    draft = q.shape[1]
    _cuda("S_committed", S_committed, torch.float32)
    code, _, _ = _projections(q, k, v, g, beta, (Lr, draft, B, H))
    _cuda("n_accepted", n_accepted, torch.int32, (B,))
    if S_new is None:
        S_new = torch.empty_like(S_committed)
    if out is None:
        out = torch.empty((Lr, B, H, draft, dv), device=S_committed.device, dtype=q.dtype)
    _cuda("S_new", S_new, torch.float32, (Lr, B, H, dk, dv))
    _cuda("out", out, q.dtype, (Lr, B, H, draft, dv))
    _check(_lib.kda_verify_replay_layers(Lr, _ptr(S_committed), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                         _ptr(beta), _ptr(n_accepted), _ptr(S_new), _ptr(out), draft,
                                         B, H, dk, dv, code, mode, _stream(stream, S_committed.device)),
           "kda_verify_replay_layers")
    return S_new, out


def _state_dims(layout, dk, dv):
    if layout == LAYOUT_KV:
        return dk, dv
    if layout == LAYOUT_VK:
        return dv, dk
    raise ValueError(f"layout must be LAYOUT_KV or LAYOUT_VK, got {layout}")


def kda_decode_step_slots(S_pool, slot_ids, q, k, v, g, beta, o=None, layout=LAYOUT_KV,
                          mode=DECAY_FIRST, stream=None):
    """kda_decode_step on a slot pool, in place.

    S_pool (n_slots,H,dk,dv) for LAYOUT_KV or (n_slots,H,dv,dk) for LAYOUT_VK, fp32;
    slot_ids int32 (B,): row b updates slot slot_ids[b] (ids outside [0, n_slots) skip the
    row, whose output is zero). Projections (B,H,D). Returns o (B,H,dv).
    """
    B, H, dk = q.shape
    dv = v.shape[-1]
    n_slots = S_pool.shape[0]
    _cuda("S_pool", S_pool, torch.float32, (n_slots, H, *_state_dims(layout, dk, dv)))
    _cuda("slot_ids", slot_ids, torch.int32, (B,))
    code, _, _ = _projections(q, k, v, g, beta, (B, H))
    if o is None:
        o = torch.empty((B, H, dv), device=q.device, dtype=q.dtype)
    _cuda("o", o, q.dtype, (B, H, dv))
    _check(_lib.kda_decode_step_slots(_ptr(S_pool), n_slots, _ptr(slot_ids), layout, _ptr(q), _ptr(k),
                                      _ptr(v), _ptr(g), _ptr(beta), _ptr(o), B, H, dk, dv, code, mode,
                                      _stream(stream, q.device)),
           "kda_decode_step_slots")
    return o


def kda_verify_replay_slots(S_pool, q, k, v, g, beta, n_accepted, slot_in, slot_out=None,
                            S_pool_new=None, out=None, layout=LAYOUT_KV, mode=DECAY_FIRST, stream=None):
    """kda_verify_replay_layers on slot pools.

    S_pool (L,n_slots,H,<state>) fp32 with <state> (dk,dv) for LAYOUT_KV, (dv,dk) for
    LAYOUT_VK; projections (L,draft,B,H,D); n_accepted, slot_in, slot_out int32 (B,).
    Row b of layer l reads slot slot_in[b] of S_pool and writes slot slot_out[b]
    (slot_in when None) of S_pool_new, which may be S_pool itself when slot_out names
    other slots. Returns (S_pool_new, out (L,B,H,draft,dv)).
    """
    Lr, draft, B, H, dk = q.shape
    dv = v.shape[-1]
    n_slots = S_pool.shape[1]
    shape = (Lr, n_slots, H, *_state_dims(layout, dk, dv))
    _cuda("S_pool", S_pool, torch.float32, shape)
    code, _, _ = _projections(q, k, v, g, beta, (Lr, draft, B, H))
    _cuda("n_accepted", n_accepted, torch.int32, (B,))
    _cuda("slot_in", slot_in, torch.int32, (B,))
    if slot_out is not None:
        _cuda("slot_out", slot_out, torch.int32, (B,))
    if S_pool_new is None:
        S_pool_new = torch.zeros_like(S_pool)
    _cuda("S_pool_new", S_pool_new, torch.float32, shape)
    if out is None:
        out = torch.empty((Lr, B, H, draft, dv), device=q.device, dtype=q.dtype)
    _cuda("out", out, q.dtype, (Lr, B, H, draft, dv))
    _check(_lib.kda_verify_replay_slots(Lr, _ptr(S_pool), _ptr(S_pool_new), n_slots, _ptr(slot_in),
                                        _ptr(slot_out), layout, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(n_accepted), _ptr(out), draft, B, H, dk, dv,
                                        code, mode, _stream(stream, q.device)),
           "kda_verify_replay_slots")
    return S_pool_new, out


class RawInputRing:
    """Device window of raw draft projections replayed at commit (kda_ring_* entry points).

    Owns a CUDA uint8 arena of kda_ring_bytes(...) bytes; push() copies one step's
    (q, k, v, g, beta) of shapes (B,H,dk) / (B,H,dv) / (B,H) in, overwriting the oldest
    step once `capacity` are held; window() returns the held steps oldest first as
    (len,B,H,D) tensors; verify_replay() replays the accepted prefix in place.
    """

    def __init__(self, capacity, B, H, dk, dv, dtype=torch.float32, device="cuda"):
        self.B, self.H, self.dk, self.dv, self.dtype = B, H, dk, dv, dtype
        code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
        n = _lib.kda_ring_bytes(capacity, B, H, dk, dv, code)
        if n < 0:
            _check(int(n), "kda_ring_bytes")
        self.arena = torch.empty(int(n), dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        _check(_lib.kda_ring_create(ctypes.c_void_p(self.arena.data_ptr()), capacity, B, H, dk, dv, code,
                                    ctypes.byref(h)), "kda_ring_create")
        self._h = h
        self.capacity = capacity

    def __del__(self):
        if getattr(self, "_h", None):
            _lib.kda_ring_destroy(self._h)
            self._h = None

    def __len__(self):
        return int(_lib.kda_ring_len(self._h))

    def reset(self):
        _check(_lib.kda_ring_reset(self._h), "kda_ring_reset")

    def push(self, q, k, v, g, beta, stream=None):
        for nm, t, shp in (("q", q, (self.B, self.H, self.dk)), ("k", k, (self.B, self.H, self.dk)),
                           ("g", g, (self.B, self.H, self.dk)), ("v", v, (self.B, self.H, self.dv)),
                           ("beta", beta, (self.B, self.H))):
            _cuda(nm, t, self.dtype, shp)
        _check(_lib.kda_ring_push(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _stream(stream, self.arena.device)), "kda_ring_push")

    def window(self, stream=None):
        n = len(self)
        dev = self.arena.device
        q = torch.empty((n, self.B, self.H, self.dk), dtype=self.dtype, device=dev)
        k, g = torch.empty_like(q), torch.empty_like(q)
        v = torch.empty((n, self.B, self.H, self.dv), dtype=self.dtype, device=dev)
        beta = torch.empty((n, self.B, self.H), dtype=self.dtype, device=dev)
        _check(_lib.kda_ring_window(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    _stream(stream, dev)), "kda_ring_window")
        return q, k, v, g, beta

    def verify_replay(self, S_committed, n_accepted, S_new=None, out=None, mode=DECAY_FIRST, stream=None):
        n = len(self)
        _cuda("S_committed", S_committed, torch.float32, (self.B, self.H, self.dk, self.dv))
        _cuda("n_accepted", n_accepted, torch.int32, (self.B,))
        if S_new is None:
            S_new = torch.empty_like(S_committed)
        if out is None:
            out = torch.empty((self.B, self.H, n, self.dv), dtype=self.dtype, device=S_committed.device)
        _cuda("S_new", S_new, torch.float32, (self.B, self.H, self.dk, self.dv))
        _cuda("out", out, self.dtype, (self.B, self.H, n, self.dv))
        _check(_lib.kda_verify_replay_ring(self._h, _ptr(S_committed), _ptr(n_accepted), _ptr(S_new), _ptr(out),
                                           mode, _stream(stream, S_committed.device)), "kda_verify_replay_ring")
        return S_new, out


def _cu_array(cu_seqlens: Optional[Sequence[int]]):
    if cu_seqlens is None:
        return None, 1
    arr = (ctypes.c_int32 * len(cu_seqlens))(*[int(x) for x in cu_seqlens])
    return arr, len(cu_seqlens) - 1


def kda_num_checkpoints(cu_seqlens, T, ckpt_stride) -> int:
    arr, n = _cu_array(cu_seqlens)
    r = _lib.kda_num_checkpoints(arr, n, int(T), int(ckpt_stride))
    if r < 0:
        _check(int(r), "kda_num_checkpoints")
    return int(r)


def kda_prefill_workspace_bytes(cu_seqlens, T, H, dk, dv, dtype) -> int:
    arr, n = _cu_array(cu_seqlens)
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    r = _lib.kda_prefill_workspace_bytes(arr, n, int(T), int(H), int(dk), int(dv), code)
    if r < 0:
        _check(int(r), "kda_prefill_workspace_bytes")
    return int(r)


def kda_device_errors() -> int:
    """Read and clear the device error word (DEVERR_WAIT: an mbarrier wait timed out;
    DEVERR_GATE: a chunked prefill read a gate outside [-10, 0] or a NaN gate)."""
    flags = ctypes.c_int(0)
    _check(_lib.kda_device_errors(ctypes.byref(flags)), "kda_device_errors")
    return int(flags.value)


def kda_set_prefill_chain_columns(cols: int) -> None:
    """State columns per chain CTA of the tensor-core prefill: 32, 64, or 0 (chosen per call)."""
    _check(_lib.kda_set_prefill_chain_columns(int(cols)), "kda_set_prefill_chain_columns")


def kda_input_prep(mixed, conv_weight, g_logits, beta_logits, cu_seqlens=None, window_in=None,
                   window_out=None, g_min=-5.0, act=ACT_SILU, ckpt_stride=0, conv_ckpt=None, out=None,
                   stream=None):
    """Input prologue for prefill: ShortConv + activation + L2Norm of q, k + gates from logits.

    mixed (T, H*(2dk+dv)) rows [q | k | v]; conv_weight (C, w); g_logits (T,H,dk);
    beta_logits (T,H); window_in / window_out (N, w-1, C) or None; conv_ckpt
    (num_ckpt, w-1, C) or None (needs ckpt_stride). out: optional dict of q,k,v,g,beta.
    Returns dict q, k, g (T,H,dk), v (T,H,dv), beta (T,H) in mixed's dtype.
    """
    T, C = mixed.shape
    H, dk = g_logits.shape[1], g_logits.shape[2]
    dv = C // H - 2 * dk
    if dv <= 0 or H * (2 * dk + dv) != C:
        raise ValueError(f"mixed width {C} does not split as H*(2*dk+dv) with H={H}, dk={dk}")
    dt = mixed.dtype
    code = _dtype_code(mixed)
    w = conv_weight.shape[1]
    arr, N = _cu_array(cu_seqlens)
    _cuda("mixed", mixed, dt)
    _cuda("conv_weight", conv_weight, dt, (C, w))
    _cuda("g_logits", g_logits, dt, (T, H, dk))
    _cuda("beta_logits", beta_logits, dt, (T, H))
    for name, t in (("window_in", window_in), ("window_out", window_out)):
        if t is not None:
            _cuda(name, t, dt, (N, w - 1, C))
    n_ck = 0
    if conv_ckpt is not None:
        n_ck = conv_ckpt.shape[0]
        _cuda("conv_ckpt", conv_ckpt, dt, (n_ck, w - 1, C))
    if out is None:
        dev = mixed.device
        out = {"q": torch.empty(T, H, dk, dtype=dt, device=dev), "k": torch.empty(T, H, dk, dtype=dt, device=dev),
               "v": torch.empty(T, H, dv, dtype=dt, device=dev), "g": torch.empty(T, H, dk, dtype=dt, device=dev),
               "beta": torch.empty(T, H, dtype=dt, device=dev)}
    for n, shp in (("q", (T, H, dk)), ("k", (T, H, dk)), ("v", (T, H, dv)), ("g", (T, H, dk)), ("beta", (T, H))):
        _cuda(n, out[n], dt, shp)
    _check(_lib.kda_input_prep(_ptr(mixed), _ptr(conv_weight), w, _ptr(window_in), _ptr(window_out),
                               _ptr(g_logits), _ptr(beta_logits), float(g_min), act, arr, N, T, H, dk, dv, code,
                               _ptr(out["q"]), _ptr(out["k"]), _ptr(out["v"]), _ptr(out["g"]), _ptr(out["beta"]),
                               int(ckpt_stride), _ptr(conv_ckpt), n_ck, _stream(stream, mixed.device)),
           "kda_input_prep")
    return out


def kda_decode_step_fused(S, conv_state, mixed, conv_weight, g_logits, beta_logits, o=None, slot_ids=None,
                          layout=LAYOUT_KV, g_min=-5.0, act=ACT_SILU, keep_projections=False,
                          mode=DECAY_FIRST, stream=None):
    """One decode token with the input prologue fused in; S and conv_state updated in place.

    S (B or n_slots, H, <state>) fp32; conv_state (B or n_slots, w-1, C); mixed (B, C);
    conv_weight (C, w); g_logits (B,H,dk); beta_logits (B,H); slot_ids int32 (B,) or None.
    Returns o (B,H,dv), or (o, dict of the prepared q,k,v,g,beta) with keep_projections.
    """
    B, H, dk = g_logits.shape
    C = mixed.shape[1]
    dv = C // H - 2 * dk
    dt = mixed.dtype
    code = _dtype_code(mixed)
    w = conv_weight.shape[1]
    rows = S.shape[0]
    _cuda("S", S, torch.float32, (rows, H, *_state_dims(layout, dk, dv)))
    _cuda("conv_state", conv_state, dt, (rows, w - 1, C))
    _cuda("mixed", mixed, dt, (B, C))
    _cuda("conv_weight", conv_weight, dt, (C, w))
    _cuda("g_logits", g_logits, dt, (B, H, dk))
    _cuda("beta_logits", beta_logits, dt, (B, H))
    if slot_ids is not None:
        _cuda("slot_ids", slot_ids, torch.int32, (B,))
    elif rows != B:
        raise ValueError(f"S has {rows} rows for a batch of {B} and no slot_ids")
    if o is None:
        o = torch.empty(B, H, dv, dtype=dt, device=mixed.device)
    _cuda("o", o, dt, (B, H, dv))
    kept = None
    if keep_projections:
        dev = mixed.device
        kept = {"q": torch.zeros(B, H, dk, dtype=dt, device=dev), "k": torch.zeros(B, H, dk, dtype=dt, device=dev),
                "v": torch.zeros(B, H, dv, dtype=dt, device=dev), "g": torch.zeros(B, H, dk, dtype=dt, device=dev),
                "beta": torch.zeros(B, H, dtype=dt, device=dev)}
    kp = kept or {}
    _check(_lib.kda_decode_step_fused(_ptr(S), rows, _ptr(slot_ids), layout, _ptr(conv_state), _ptr(mixed),
                                      _ptr(conv_weight), w, _ptr(g_logits), _ptr(beta_logits), float(g_min), act,
                                      _ptr(o), _ptr(kp.get("q")), _ptr(kp.get("k")), _ptr(kp.get("v")),
                                      _ptr(kp.get("g")), _ptr(kp.get("beta")), B, H, dk, dv, code, mode,
                                      _stream(stream, mixed.device)),
           "kda_decode_step_fused")
    return (o, kept) if keep_projections else o


def kda_prefill_chunked(S0, q, k, v, g, beta, cu_seqlens=None, chunk=64, ckpt_stride=512,
                        o=None, S_final=None, page_pool=None, ckpt_page_ids=None, ckpt_pos=None,
                        mode=DECAY_FIRST, stream=None, workspace="auto"):
    """Chunked prefill of packed sequences with chunk-aligned checkpoints.

    q,k,g (T,H,dk); v (T,H,dv); beta (T,H); cu_seqlens: host list of N+1 ints (None: one
    sequence). S0 (N,H,dk,dv) fp32 or None (zero state). page_pool: a PagePool (or None
    when no checkpoints are emitted); ckpt_page_ids: CUDA int32 tensor with one page per
    checkpoint. workspace: "auto" (allocate what the tensor-core kernels need), None (no
    workspace: the fp32 CUDA-core kernel runs) or a CUDA uint8 tensor. Returns (o, S_final).
    """
    T, Hq, dk = q.shape
    code, _, dv = _projections(q, k, v, g, beta, (T, Hq))
    arr, N = _cu_array(cu_seqlens)
    dev = q.device
    if S0 is not None:
        _cuda("S0", S0, torch.float32, (N, Hq, dk, dv))
    if o is None:
        o = torch.empty((T, Hq, dv), device=dev, dtype=q.dtype)
    if S_final is None:
        S_final = torch.empty((N, Hq, dk, dv), device=dev, dtype=torch.float32)
    _cuda("o", o, q.dtype, (T, Hq, dv))
    _cuda("S_final", S_final, torch.float32, (N, Hq, dk, dv))
    base, page_bytes, n_ck = None, 0, 0
    if ckpt_page_ids is not None:
        _cuda("ckpt_page_ids", ckpt_page_ids, torch.int32)
        n_ck = ckpt_page_ids.numel()
        if page_pool is None:
            raise ValueError("ckpt_page_ids given without a page_pool")
        base, page_bytes = ctypes.c_void_p(page_pool.arena.data_ptr()), page_pool.page_bytes
    if ckpt_pos is not None:
        _cuda("ckpt_pos", ckpt_pos, torch.int32)
    if isinstance(workspace, str):
        need = kda_prefill_workspace_bytes(cu_seqlens, T, Hq, dk, dv, q.dtype)
        workspace = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
    ws_bytes = 0
    if workspace is not None:
        _cuda("workspace", workspace, torch.uint8)
        ws_bytes = workspace.numel()
    _check(_lib.kda_prefill_chunked(_ptr(S0), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    arr, N, T, Hq, dk, dv, code, chunk, ckpt_stride,
                                    _ptr(o), _ptr(S_final), base, page_bytes,
                                    _ptr(ckpt_page_ids), _ptr(ckpt_pos), n_ck,
                                    _ptr(workspace), ws_bytes, mode, _stream(stream, dev)),
           "kda_prefill_chunked")
    return o, S_final


def kda_prefill_scan_workspace_bytes(T, H, dk, dv, dtype=torch.bfloat16, ckpt_stride=512, segments=0) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    r = _lib.kda_prefill_scan_workspace_bytes(int(T), int(H), int(dk), int(dv), code, int(ckpt_stride),
                                              int(segments))
    if r < 0:
        _check(int(r), "kda_prefill_scan_workspace_bytes")
    return int(r)


def kda_prefill_scan(S0, q, k, v, g, beta, chunk=64, ckpt_stride=512, o=None, S_final=None, page_pool=None,
                     ckpt_page_ids=None, ckpt_pos=None, segments=0, workspace=None, mode=DECAY_FIRST,
                     stream=None):
    """Sequence-parallel prefill of one sequence (q,k,g (T,H,dk); v (T,H,dv); beta (T,H); bf16).

    S0 (1,H,dk,dv) fp32 or None. segments: 0 = chosen from the SM count. workspace: None
    (allocated) or a CUDA uint8 tensor of kda_prefill_scan_workspace_bytes(...). Returns (o, S_final).
    """
    T, Hq, dk = q.shape
    code, _, dv = _projections(q, k, v, g, beta, (T, Hq))
    dev = q.device
    if S0 is not None:
        _cuda("S0", S0, torch.float32, (1, Hq, dk, dv))
    if o is None:
        o = torch.empty((T, Hq, dv), device=dev, dtype=q.dtype)
    if S_final is None:
        S_final = torch.empty((1, Hq, dk, dv), device=dev, dtype=torch.float32)
    _cuda("o", o, q.dtype, (T, Hq, dv))
    _cuda("S_final", S_final, torch.float32, (1, Hq, dk, dv))
    stride = ckpt_stride if page_pool is not None else 0       # no pool: no checkpoints
    n_ck = 0
    if page_pool is not None and ckpt_page_ids is not None:
        _cuda("ckpt_page_ids", ckpt_page_ids, torch.int32)
        n_ck = ckpt_page_ids.numel()
        if ckpt_pos is not None:
            _cuda("ckpt_pos", ckpt_pos, torch.int32)
    need = kda_prefill_scan_workspace_bytes(T, Hq, dk, dv, q.dtype, stride, segments)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _cuda("workspace", workspace, torch.uint8)
    _check(_lib.kda_prefill_scan(_ptr(S0), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), T, Hq, dk, dv, code,
                                 chunk, stride, _ptr(o), _ptr(S_final),
                                 ctypes.c_void_p(page_pool.arena.data_ptr()) if page_pool is not None else None,
                                 page_pool.page_bytes if page_pool is not None else 0,
                                 _ptr(ckpt_page_ids) if n_ck else None, _ptr(ckpt_pos) if n_ck else None,
                                 n_ck, _ptr(workspace), workspace.numel(), int(segments), mode,
                                 _stream(stream, dev)),
           "kda_prefill_scan")
    return o, S_final


def _host(name, t, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def kda_prefill_host_scratch_bytes(H, dk, dv, dtype, ckpt_stride=512, segment_tokens=1024) -> int:
    """Device scratch kda_prefill_chunked_host needs."""
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    n = _lib.kda_prefill_host_scratch_bytes(H, dk, dv, code, ckpt_stride, segment_tokens)
    if n < 0:
        _check(int(n), "kda_prefill_host_scratch_bytes")
    return int(n)


def kda_prefill_chunked_host(S0, q, k, v, g, beta, o, S_final, scratch, cu_seqlens=None, chunk=64,
                             ckpt_stride=512, page_pool=None, ckpt_page_ids=None, ckpt_pos=None,
                             segment_tokens=1024, mode=DECAY_FIRST, stream=None, device=None):
    """kda_prefill_chunked on host-resident tensors (pin them for the copies to overlap).

    q,k,g (T,H,dk), v (T,H,dv), beta (T,H), S0 (N,H,dk,dv) or None, o (T,H,dv) and S_final
    (N,H,dk,dv): CPU tensors. scratch: CUDA uint8 tensor of at least
    kda_prefill_host_scratch_bytes(...) bytes. Checkpoint pages, ids and positions stay on the
    device. The call returns once everything is enqueued on `stream`; synchronise it before
    reading o and S_final. Returns (o, S_final).
    """
    T, Hq, dk = q.shape
    dv = v.shape[-1]
    dt = q.dtype
    code = _dtype_code(q)
    for nm, t, shp in (("q", q, (T, Hq, dk)), ("k", k, (T, Hq, dk)), ("g", g, (T, Hq, dk)),
                       ("v", v, (T, Hq, dv)), ("beta", beta, (T, Hq))):
        _host(nm, t, dt, shp)
    arr, N = _cu_array(cu_seqlens)
    if S0 is not None:
        _host("S0", S0, torch.float32, (N, Hq, dk, dv))
    _host("o", o, dt, (T, Hq, dv))
    _host("S_final", S_final, torch.float32, (N, Hq, dk, dv))
    _cuda("scratch", scratch, torch.uint8)
    dev = scratch.device if device is None else device
    base, page_bytes, n_ck = None, 0, 0
    if ckpt_page_ids is not None:
        _cuda("ckpt_page_ids", ckpt_page_ids, torch.int32)
        n_ck = ckpt_page_ids.numel()
        if page_pool is None:
            raise ValueError("ckpt_page_ids given without a page_pool")
        base, page_bytes = ctypes.c_void_p(page_pool.arena.data_ptr()), page_pool.page_bytes
    if ckpt_pos is not None:
        _cuda("ckpt_pos", ckpt_pos, torch.int32)
    _check(_lib.kda_prefill_chunked_host(_ptr(S0), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                         arr, N, T, Hq, dk, dv, code, chunk, ckpt_stride,
                                         _ptr(o), _ptr(S_final), base, page_bytes,
                                         _ptr(ckpt_page_ids), _ptr(ckpt_pos), n_ck,
                                         _ptr(scratch), scratch.numel(), segment_tokens, mode,
                                         _stream(stream, dev)),
           "kda_prefill_chunked_host")
    return o, S_final


def kda_prefill_chunked_noalloc(S0, q, k, v, g, beta, o, S_final, cu_seqlens=None, chunk=64,
                                ckpt_stride=512, page_pool=None, ckpt_page_ids=None, ckpt_pos=None,
                                mode=DECAY_FIRST, stream=None):
    """kda_prefill_chunked for callers that cannot allocate device memory at call time.

    The outputs o and S_final must be passed in (nothing is allocated here, on the
    host side of the binding either); the tensor-core scratch is the library's
    fixed built-in device array, so a call needing more than it holds is refused.
    """
    T, Hq, dk = q.shape
    code, _, dv = _projections(q, k, v, g, beta, (T, Hq))
    arr, N = _cu_array(cu_seqlens)
    if S0 is not None:
        _cuda("S0", S0, torch.float32, (N, Hq, dk, dv))
    _cuda("o", o, q.dtype, (T, Hq, dv))
    _cuda("S_final", S_final, torch.float32, (N, Hq, dk, dv))
    base, page_bytes, n_ck = None, 0, 0
    if ckpt_page_ids is not None:
        _cuda("ckpt_page_ids", ckpt_page_ids, torch.int32)
        n_ck = ckpt_page_ids.numel()
        base, page_bytes = ctypes.c_void_p(page_pool.arena.data_ptr()), page_pool.page_bytes
    _check(_lib.kda_prefill_chunked_noalloc(_ptr(S0), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                            arr, N, T, Hq, dk, dv, code, chunk, ckpt_stride,
                                            _ptr(o), _ptr(S_final), base, page_bytes,
                                            _ptr(ckpt_page_ids), _ptr(ckpt_pos), n_ck, mode,
                                            _stream(stream, q.device)),
           "kda_prefill_chunked_noalloc")
    return o, S_final


def kda_pack_heads(S, flat=None, flat_elems=None, stream=None):
    """(B,H,dk,dv) fp32 (the (b,h) dims may be strided) -> flat fp32, zero-padded."""
    if not S.is_cuda or S.dtype != torch.float32:
        raise TypeError("S must be a CUDA float32 tensor")
    B, H, dk, dv = S.shape
    if S.stride(3) != 1 or S.stride(2) != dv:
        raise ValueError("each (dk, dv) block of S must be contiguous")
    n = B * H * dk * dv
    if flat is None:
        flat = torch.empty(flat_elems or n, device=S.device, dtype=torch.float32)
    _cuda("flat", flat, torch.float32)
    _check(_lib.kda_pack_heads(_ptr(S), S.stride(0), S.stride(1), _ptr(flat), flat.numel(),
                               B, H, dk, dv, _stream(stream, S.device)), "kda_pack_heads")
    return flat


def kda_unpack_heads(flat, S, stream=None):
    """flat fp32 -> S (B,H,dk,dv), written in place (the (b,h) dims may be strided)."""
    _cuda("flat", flat, torch.float32)
    if not S.is_cuda or S.dtype != torch.float32:
        raise TypeError("S must be a CUDA float32 tensor")
    B, H, dk, dv = S.shape
    if S.stride(3) != 1 or S.stride(2) != dv:
        raise ValueError("each (dk, dv) block of S must be contiguous")
    if flat.numel() < B * H * dk * dv:
        raise ValueError("flat is smaller than the state")
    _check(_lib.kda_unpack_heads(_ptr(flat), _ptr(S), S.stride(0), S.stride(1), B, H, dk, dv,
                                 _stream(stream, S.device)), "kda_unpack_heads")
    return S


def kda_snapshot_cost_ratio(H, dk, dv) -> float:
    r = _lib.kda_snapshot_cost_ratio(int(H), int(dk), int(dv))
    if r < 0:
        raise ValueError(_lib.kda_last_error().decode())
    return r


class PagePool:
    """Unified page pool: a device arena (owned by PyTorch) plus the library's host free list.

    One free list hands out pages of both kinds (KDA state, MLA KV), lowest index first.
    """

    def __init__(self, page_bytes: int, n_pages: int, device="cuda"):
        self.page_bytes = int(page_bytes)
        self.n_pages = int(n_pages)
        self.arena = torch.empty(self.page_bytes * self.n_pages, dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        _check(_lib.kda_pool_create(ctypes.c_void_p(self.arena.data_ptr()), self.page_bytes,
                                    self.n_pages, ctypes.byref(h)), "kda_pool_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.kda_pool_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def alloc(self, n: int, kind: int = PAGE_KDA_STATE):
        ids = (ctypes.c_int32 * max(int(n), 1))()
        _check(_lib.kda_pool_alloc(self._h, kind, int(n), ids), "kda_pool_alloc")
        return [int(ids[i]) for i in range(int(n))]

    def free(self, ids):
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check(_lib.kda_pool_free(self._h, len(ids), arr), "kda_pool_free")

    def num_free(self) -> int:
        return int(_lib.kda_pool_num_free(self._h))

    def kind(self, page_id: int) -> int:
        return int(_lib.kda_pool_page_kind(self._h, int(page_id)))

    def page(self, page_id: int, dtype=torch.float32) -> torch.Tensor:
        """View of one page's bytes as a 1-D tensor (no copy)."""
        off = int(page_id) * self.page_bytes
        return self.arena[off:off + self.page_bytes].view(dtype)

    def store_kda(self, page_id: int, S: torch.Tensor, stream=None):
        B, H, dk, dv = S.shape
        _check(_lib.kda_store_kda(self._h, int(page_id), _ptr(S), S.stride(0), S.stride(1),
                                  B, H, dk, dv, _stream(stream, S.device)), "kda_store_kda")

    def load_kda(self, page_id: int, S: torch.Tensor, stream=None):
        B, H, dk, dv = S.shape
        _check(_lib.kda_load_kda(self._h, int(page_id), _ptr(S), S.stride(0), S.stride(1),
                                 B, H, dk, dv, _stream(stream, S.device)), "kda_load_kda")
        return S
