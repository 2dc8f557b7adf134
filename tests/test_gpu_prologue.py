"""GPU parity of the input prologue (kda_input_prep, kda_decode_step_fused) against the
fp64 oracle: ShortConv with the carried window, activation, per-head L2Norm of q and k,
gates from logits, the window after each sequence and the conv checkpoints (raw rows:
bit-exact), and the fused decode step that runs the prologue and one recurrence step."""
import numpy as np
import pytest
import torch

from kda_delta_rule_gb300 import inputs as I
from oracle import kda_oracle as O
from parity import TOL_BF16_OUT, TOL_BF16_STATE, TOL_BF16_STORED_OUT, TOL_F32, rel

pytestmark = pytest.mark.gpu
f = I.to_f64_numpy
G_MIN = -5.0


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


def _tol(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16_STORED_OUT


def _oracle_prep(p, cu, H, dk, dv, act, n_ck_stride=0):
    """Per sequence: oracle prologue outputs concatenated, windows after, conv checkpoints."""
    outs = {n: [] for n in ("q", "k", "v", "g", "beta")}
    wins, cks = [], []
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        win = f(p["window"][n])
        q, k, v, g, beta, wo = O.input_prep(f(p["mixed"][a:b]), f(p["weight"]), win, f(p["g_logits"][a:b]),
                                            f(p["beta_logits"][a:b]), H, dk, dv, G_MIN, act)
        for name, val in zip(("q", "k", "v", "g", "beta"), (q, k, v, g, beta)):
            outs[name].append(val)
        wins.append(wo)
        if n_ck_stride:
            for j in range(1, (b - a) // n_ck_stride + 1):
                cks.append(O.conv_window_at(f(p["mixed"][a:b]), win, j * n_ck_stride))
    return {n: np.concatenate(v) for n, v in outs.items()}, np.stack(wins), cks


@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv,w", [(128, 128, 4), (64, 32, 2), (32, 128, 8), (128, 64, 3)])
def test_input_prep_varlen(K, dk, dv, w, dtype, act):
    """Sequences shorter than the window, ragged tiles, an empty sequence, carried windows,
    conv checkpoints every 64 tokens."""
    H, lengths, stride = 2, [2, 37, 0, 200, 64, 129], 64
    p, cu = I.prologue_inputs(lengths, H, dk, dv, w=w, dtype=dtype, seed=dk + dv + w + act)
    pd = {n: t.cuda() for n, t in p.items()}
    n_ck = K.kda_num_checkpoints(cu, cu[-1], stride)
    C = H * (2 * dk + dv)
    win_out = torch.full((len(lengths), w - 1, C), 7.0, dtype=dtype, device="cuda")
    ck = torch.full((n_ck, w - 1, C), 7.0, dtype=dtype, device="cuda")
    out = K.kda_input_prep(pd["mixed"], pd["weight"], pd["g_logits"], pd["beta_logits"], cu_seqlens=cu,
                           window_in=pd["window"], window_out=win_out, g_min=G_MIN, act=act,
                           ckpt_stride=stride, conv_ckpt=ck)
    ref, wins, cks = _oracle_prep(p, cu, H, dk, dv, act, stride)
    torch.cuda.synchronize()
    for n in ("q", "k", "v", "g", "beta"):
        assert rel(out[n], ref[n]) < _tol(dtype), n
    # windows and conv checkpoints are raw rows: exact copies
    assert np.array_equal(f(win_out), wins)
    assert len(cks) == n_ck and np.array_equal(f(ck), np.stack(cks))


def test_input_prep_zero_window_and_single_sequence(K):
    """No window given (a fresh sequence: zeros), cu_seqlens None, T not a multiple of 32."""
    H, dk, dv, w, T = 3, 64, 64, 4, 333
    p, cu = I.prologue_inputs([T], H, dk, dv, w=w, dtype=torch.float32, seed=5, zero_window=True)
    pd = {n: t.cuda() for n, t in p.items()}
    out = K.kda_input_prep(pd["mixed"], pd["weight"], pd["g_logits"], pd["beta_logits"], g_min=G_MIN)
    ref, _, _ = _oracle_prep(p, cu, H, dk, dv, 1)
    torch.cuda.synchronize()
    for n in ("q", "k", "v", "g", "beta"):
        assert rel(out[n], ref[n]) < TOL_F32, n


def test_input_prep_then_prefill_matches_oracle(K):
    """Prologue then the tensor-core prefill: two sequences, checkpoints every 512 tokens."""
    H, dk, dv, w = 4, 128, 128, 4
    lengths = [1100, 700]
    p, cu = I.prologue_inputs(lengths, H, dk, dv, w=w, dtype=torch.bfloat16, seed=21)
    pd = {n: t.cuda() for n, t in p.items()}
    S0, _, _ = I.prefill_inputs(lengths, H, dk, dv, dtype=torch.bfloat16, seed=22)
    proj = K.kda_input_prep(pd["mixed"], pd["weight"], pd["g_logits"], pd["beta_logits"], cu_seqlens=cu,
                            window_in=pd["window"], g_min=G_MIN)
    o, S_f = K.kda_prefill_chunked(S0.cuda(), proj["q"], proj["k"], proj["v"], proj["g"], proj["beta"],
                                   cu_seqlens=cu, ckpt_stride=0)
    torch.cuda.synchronize()
    # oracle: its own prologue on the raw inputs, then the recurrence from the stored
    # (bf16) projections the GPU produced is not used: the chain below is all oracle
    ref, _, _ = _oracle_prep(p, cu, H, dk, dv, 1)
    o_ref, S_ref = [], []
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        on, Sn = O.kda_recurrent(f(S0[n]), *(ref[x][a:b] for x in ("q", "k", "v", "g", "beta")))
        o_ref.append(on)
        S_ref.append(Sn)
    assert rel(o, np.concatenate(o_ref)) < TOL_BF16_OUT
    assert rel(S_f, np.stack(S_ref)) < TOL_BF16_STATE


def _fused_oracle(S, win, mixed, weight, gl, bl, H, dk, dv, act, mode=0):
    """Oracle for one fused decode token of one batch row: prologue of one token, one step."""
    q, k, v, g, beta, wo = O.input_prep(mixed[None], weight, win, gl[None], bl[None], H, dk, dv, G_MIN, act)
    o, S_new = O.kda_step(S, q[0], k[0], v[0], g[0], beta[0], mode)
    return o, S_new, wo, (q[0], k[0], v[0], g[0], beta[0])


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(128, 128), (32, 64), (64, 32), (128, 32)])
def test_decode_fused_matches_oracle(K, dk, dv, dtype, mode):
    B, H, w = 3, 4, 4
    p, _ = I.prologue_inputs([1] * B, H, dk, dv, w=w, dtype=dtype, seed=dk * 3 + dv + mode)
    S, _ = I.decode_inputs(B, H, dk, dv, dtype=dtype, seed=dk + dv)
    Sd = S.cuda()
    win = p["window"].cuda().clone()
    o, kept = K.kda_decode_step_fused(Sd, win, p["mixed"].cuda(), p["weight"].cuda(), p["g_logits"].cuda(),
                                      p["beta_logits"].cuda(), g_min=G_MIN, keep_projections=True, mode=mode)
    torch.cuda.synchronize()
    for b in range(B):
        o_r, S_r, w_r, pr = _fused_oracle(f(S[b]), f(p["window"][b]), f(p["mixed"][b]), f(p["weight"]),
                                          f(p["g_logits"][b]), f(p["beta_logits"][b]), H, dk, dv, 1, mode)
        assert rel(Sd[b], S_r) < TOL_F32
        assert rel(o[b], o_r) < _tol(dtype)
        assert np.array_equal(f(win[b]), w_r)
        for name, val in zip(("q", "k", "v", "g", "beta"), pr):
            assert rel(kept[name][b], val) < _tol(dtype), name


def test_decode_fused_slots_transposed_and_padding(K):
    """Transposed pool with slot ids, one padded row: untouched slots and windows stay bitwise."""
    B, H, dk, dv, w, n_slots = 4, 2, 64, 128, 3, 9
    p, _ = I.prologue_inputs([1] * B, H, dk, dv, w=w, dtype=torch.bfloat16, seed=77)
    gen = torch.Generator().manual_seed(78)
    S_math = 0.1 * torch.randn(n_slots, H, dk, dv, generator=gen)
    pool = S_math.transpose(-1, -2).contiguous().cuda()
    C = H * (2 * dk + dv)
    wins = torch.randn(n_slots, w - 1, C, generator=gen).to(torch.bfloat16).cuda()
    slots = torch.tensor([5, -1, 0, 7], dtype=torch.int32)
    pool0, wins0 = pool.clone(), wins.clone()
    o = K.kda_decode_step_fused(pool, wins, p["mixed"].cuda(), p["weight"].cuda(), p["g_logits"].cuda(),
                                p["beta_logits"].cuda(), slot_ids=slots.cuda(), layout=K.LAYOUT_VK, g_min=G_MIN)
    torch.cuda.synchronize()
    for b in range(B):
        sl = int(slots[b])
        if sl < 0:
            assert torch.count_nonzero(o[b]) == 0
            continue
        o_r, S_r, w_r, _ = _fused_oracle(f(S_math[sl]), f(wins0[sl]), f(p["mixed"][b]), f(p["weight"]),
                                         f(p["g_logits"][b]), f(p["beta_logits"][b]), H, dk, dv, 1)
        assert rel(pool[sl].transpose(-1, -2), S_r) < TOL_F32
        assert rel(o[b], o_r) < TOL_BF16_STORED_OUT
        assert np.array_equal(f(wins[sl]), w_r)
    kept = [s for s in range(n_slots) if s not in (5, 0, 7)]
    assert torch.equal(pool[kept], pool0[kept]) and torch.equal(wins[kept], wins0[kept])


def test_decode_fused_steps_equal_prefill_prologue(K):
    """Five fused decode tokens = the prologue over the same five rows, then the recurrence."""
    B, H, dk, dv, w, T = 2, 2, 128, 128, 4, 5
    p, cu = I.prologue_inputs([T] * B, H, dk, dv, w=w, dtype=torch.float32, seed=91)
    S, _ = I.decode_inputs(B, H, dk, dv, dtype=torch.float32, seed=92)
    Sd = S.cuda()
    win = p["window"].cuda().clone()
    mixed = p["mixed"].view(B, T, -1)
    gl = p["g_logits"].view(B, T, H, dk)
    bl = p["beta_logits"].view(B, T, H)
    outs = []
    for t in range(T):
        outs.append(K.kda_decode_step_fused(Sd, win, mixed[:, t].contiguous().cuda(), p["weight"].cuda(),
                                            gl[:, t].contiguous().cuda(), bl[:, t].contiguous().cuda(),
                                            g_min=G_MIN))
    torch.cuda.synchronize()
    ref, wins, _ = _oracle_prep(p, cu, H, dk, dv, 1)
    for b in range(B):
        sl = slice(cu[b], cu[b + 1])
        o_r, S_r = O.kda_recurrent(f(S[b]), *(ref[x][sl] for x in ("q", "k", "v", "g", "beta")))
        assert rel(torch.stack([o[b] for o in outs]), o_r) < TOL_F32
        assert rel(Sd[b], S_r) < TOL_F32
        assert np.array_equal(f(win[b]), wins[b])
