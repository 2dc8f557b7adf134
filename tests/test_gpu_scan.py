"""GPU parity of the sequence-parallel prefill (kda_prefill_scan) against the fp64 oracle:
outputs, final state, checkpoint pages and positions of one long sequence cut into segments
(first piece from S0, middle pieces' local states and transitions, fp32 scan of the starts,
remaining pieces from their starts)."""
import numpy as np
import pytest
import torch

from kda_delta_rule_gb300 import inputs as I
from oracle import kda_oracle as O
from parity import TOL_BF16_OUT, TOL_BF16_STATE, rel

pytestmark = pytest.mark.gpu
f = I.to_f64_numpy


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


def _scan(K, T, H, dv, stride, segments, mode=0, seed=0, S0_none=False):
    dk = 128
    S0, p, cu = I.prefill_inputs([T], H, dk, dv, dtype=torch.bfloat16, seed=seed)
    n_ck = K.kda_num_checkpoints(cu, T, stride) if stride else 0
    page_bytes = H * dk * dv * 4 + 64
    pool = K.PagePool(page_bytes, max(n_ck, 1))
    if n_ck:
        pool.arena.fill_(0xAB)
    ids = torch.tensor(pool.alloc(n_ck)[::-1] if n_ck else [], dtype=torch.int32, device="cuda")
    pos = torch.full((n_ck,), -1, dtype=torch.int32, device="cuda")
    pd = {n: t.cuda() for n, t in p.items()}
    S0d = None if S0_none else S0.cuda()
    o, S_f = K.kda_prefill_scan(S0d, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"], ckpt_stride=stride,
                                page_pool=pool if n_ck else None, ckpt_page_ids=ids if n_ck else None,
                                ckpt_pos=pos if n_ck else None, segments=segments, mode=mode)
    torch.cuda.synchronize()
    assert K.kda_device_errors() == 0
    S0_ref = np.zeros((1, H, dk, dv)) if S0_none else f(S0)
    o_ref, S_ref, ck_ref = O.prefill_recurrent(S0_ref, *(f(p[n]) for n in ("q", "k", "v", "g", "beta")),
                                               ckpt_stride=stride, mode=mode)
    assert rel(o, o_ref) < TOL_BF16_OUT
    assert rel(S_f, S_ref) < TOL_BF16_STATE
    assert pos.tolist() == [t for _, t, _ in ck_ref]
    n_state = H * dk * dv
    for c, (_, t, st) in enumerate(ck_ref):
        page = pool.page(int(ids[c]))
        assert rel(page[:n_state].reshape(H, dk, dv), st) < TOL_BF16_STATE
        assert torch.count_nonzero(page[n_state:]) == 0
    return o, S_f


@pytest.mark.parametrize("segments", [3, 4, 8, 0])
def test_scan_matches_oracle(K, segments):
    """4 heads, 4096 tokens, checkpoints every 512: 3, 4, 8 and the chosen number of pieces."""
    _scan(K, 4096, 4, 128, 512, segments, seed=segments)


@pytest.mark.parametrize("mode", [0, 1])
def test_scan_dv64_ragged_tail_no_checkpoints(K, mode):
    """dv = 64 (one transition column block per 64 columns: two per transition), a ragged
    last piece, no checkpoints (pieces of whole 64-token chunks), zero start state."""
    _scan(K, 3000, 2, 64, 0, 5, mode=mode, seed=11, S0_none=True)


def test_scan_with_few_segments_is_the_plain_chain(K):
    """Fewer than three pieces runs the ordinary chain: the same bits as kda_prefill_chunked."""
    T, H, dk, dv = 1536, 2, 128, 128
    S0, p, cu = I.prefill_inputs([T], H, dk, dv, dtype=torch.bfloat16, seed=5)
    pd = {n: t.cuda() for n, t in p.items()}
    o1, S1 = K.kda_prefill_scan(S0.cuda(), pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"], ckpt_stride=512,
                                segments=2)
    o2, S2 = K.kda_prefill_chunked(S0.cuda(), pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"], cu_seqlens=cu,
                                   ckpt_stride=0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


def test_scan_long_sequence_sampled_against_plain_chain(K):
    """H = 4, T = 32768: the scan and the serial chain agree within the bf16 tolerances, and
    both match the oracle on two heads' final states."""
    T, H, dk, dv = 32768, 4, 128, 128
    S0, p, cu = I.prefill_inputs([T], H, dk, dv, dtype=torch.bfloat16, seed=21, device="cuda")
    o1, S1 = K.kda_prefill_scan(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], ckpt_stride=512, segments=0)
    o2, S2 = K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu, ckpt_stride=0)
    torch.cuda.synchronize()
    assert rel(o1, o2) < TOL_BF16_OUT and rel(S1, S2) < TOL_BF16_STATE
    for h in (0, 3):
        hd = {n: f(p[n][:, h]) for n in ("q", "k", "v", "g", "beta")}
        _, S_ref = O.kda_recurrent(f(S0[0, h]), hd["q"], hd["k"], hd["v"], hd["g"], hd["beta"])
        assert rel(S1[0, h], S_ref) < TOL_BF16_STATE


def test_scan_32_heads_every_head_against_oracle(K):
    """H = 32, dk = dv = 128 (the long-prefill head count), T = 4096 cut into 4 pieces, checkpoints
    every 512: outputs, final state and every checkpoint page of every head against the fp64
    oracle, one worker process per head.  The first chain launch here has 5 pseudo-sequences x
    32 heads of CTAs (several waves), the tensor-core scan 32 x 4 CTAs."""
    from oracle_pool import prefill_chunked_per_head
    T, H, d, stride = 4096, 32, 128, 512
    S0, p, cu = I.prefill_inputs([T], H, d, d, dtype=torch.bfloat16, seed=31, device="cuda")
    n_ck = K.kda_num_checkpoints(cu, T, stride)
    pool = K.PagePool(H * d * d * 4, n_ck)
    ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device="cuda")
    pos = torch.full((n_ck,), -1, dtype=torch.int32, device="cuda")
    o, S_f = K.kda_prefill_scan(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], ckpt_stride=stride, page_pool=pool,
                                ckpt_page_ids=ids, ckpt_pos=pos, segments=4)
    torch.cuda.synchronize()
    assert K.kda_device_errors() == 0
    assert pos.tolist() == [stride * j for j in range(1, n_ck + 1)]

    def np32(t):
        return t.detach().to("cpu", torch.float32).numpy()

    ref = prefill_chunked_per_head(np32(S0), *(np32(p[n]) for n in ("q", "k", "v", "g", "beta")), cu, stride,
                                   range(H))
    pages = torch.stack([pool.page(int(ids[c])).reshape(H, d, d) for c in range(n_ck)])
    for h in range(H):
        o_ref, S_ref, ck_ref = ref[h]
        assert rel(o[:, h], o_ref[:, 0]) < TOL_BF16_OUT, h
        assert rel(S_f[0, h], S_ref[0, 0]) < TOL_BF16_STATE, h
        for c in range(n_ck):
            assert rel(pages[c, h], ck_ref[c][2][0]) < TOL_BF16_STATE, (h, c)
