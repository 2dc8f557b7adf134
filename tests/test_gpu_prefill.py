"""GPU parity of the chunked prefill (outputs, final state, checkpoints) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from kda_delta_rule_gb300 import inputs as I
from oracle import kda_oracle as O
from parity import TOL_BF16_OUT, TOL_BF16_STATE, TOL_F32, rel

pytestmark = pytest.mark.gpu
f = I.to_f64_numpy


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


def run_prefill(K, S0, p, cu, H, dk, dv, stride, mode=0, pad_bytes=0, S0_none=False):
    T = cu[-1]
    n_ck = K.kda_num_checkpoints(cu, T, stride)
    page_bytes = H * dk * dv * 4 + pad_bytes
    pool = K.PagePool(page_bytes, max(n_ck, 1))
    if n_ck:
        pool.arena.fill_(0xAB)            # garbage: the emitter must overwrite all of it
    ids = torch.tensor(pool.alloc(n_ck)[::-1] if n_ck else [], dtype=torch.int32, device="cuda")
    pos = torch.full((n_ck,), -1, dtype=torch.int32, device="cuda")
    pd = {n: t.cuda() for n, t in p.items()}
    S0d = None if S0_none else S0.cuda()
    snap = None if S0d is None else S0d.clone()
    o, S_fin = K.kda_prefill_chunked(S0d, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"],
                                     cu_seqlens=cu, ckpt_stride=stride, page_pool=pool,
                                     ckpt_page_ids=ids if n_ck else None,
                                     ckpt_pos=pos if n_ck else None, mode=mode)
    torch.cuda.synchronize()
    if snap is not None:
        assert torch.equal(S0d, snap), "S0 was written"
    return o, S_fin, pool, ids, pos


def check_against_oracle(K, lengths, H, dk, dv, dtype, stride, mode=0, seed=0, pad_bytes=0,
                         state_std=0.05, S0_none=False):
    S0, p, cu = I.prefill_inputs(lengths, H, dk, dv, dtype=dtype, seed=seed, state_std=state_std)
    if S0_none:
        S0 = torch.zeros_like(S0)
    o, S_fin, pool, ids, pos = run_prefill(K, S0, p, cu, H, dk, dv, stride, mode, pad_bytes,
                                           S0_none=S0_none)
    args = [f(S0)] + [f(p[n]) for n in ("q", "k", "v", "g", "beta")]
    o_ref, S_ref, ck_ref = O.prefill_chunked(*args, cu_seqlens=cu, chunk=64, ckpt_stride=stride,
                                             mode=mode)
    tol_o = TOL_F32 if dtype == torch.float32 else TOL_BF16_OUT
    tol_s = TOL_F32 if dtype == torch.float32 else TOL_BF16_STATE
    assert rel(o, o_ref) < tol_o
    assert rel(S_fin, S_ref) < tol_s
    assert pos.tolist() == [t for _, t, _ in ck_ref]
    n_state = H * dk * dv
    for c, (n, t, st) in enumerate(ck_ref):
        page = pool.page(int(ids[c]))
        assert rel(page[:n_state].reshape(H, dk, dv), st) < tol_s
        if pad_bytes:
            assert torch.all(page[n_state:] == 0), "page tail not zeroed"
        if t == lengths[n]:
            # the last boundary of a sequence is its final state, bit for bit
            assert torch.equal(page[:n_state].reshape(H, dk, dv), S_fin[n])
    return o, S_fin


@pytest.mark.parametrize("mode", [0, 1])
def test_oracle_scale_single_sequence(K, mode):
    """B=1, H=4, dk=dv=32, T=256, chunk 64, fp32, S0 = 0."""
    o, S_fin = check_against_oracle(K, [256], 4, 32, 32, torch.float32, 64, mode=mode,
                                    state_std=0.0, S0_none=True)
    # and against the token recurrence directly
    S0, p, cu = I.prefill_inputs([256], 4, 32, 32, dtype=torch.float32, seed=0, state_std=0.0)
    args = [f(S0)] + [f(p[n]) for n in ("q", "k", "v", "g", "beta")]
    o_rec, S_rec, _ = O.prefill_recurrent(*args, cu_seqlens=cu, ckpt_stride=0, mode=mode)
    assert rel(o, o_rec) < TOL_F32 and rel(S_fin, S_rec) < TOL_F32


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128), (32, 128)])
def test_ragged_varlen_fp32(K, dk, dv):
    lengths = [1, 63, 65, 130, 0, 200, 128]
    check_against_oracle(K, lengths, 3, dk, dv, torch.float32, 64, seed=dk + dv, pad_bytes=48)


@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_inputs(K, mode):
    check_against_oracle(K, [300, 64, 512], 2, 128, 128, torch.bfloat16, 128, mode=mode, seed=7)


def test_no_checkpoints_and_empty(K):
    check_against_oracle(K, [100, 0, 37], 2, 64, 64, torch.float32, 0, seed=3)
    check_against_oracle(K, [0, 0], 2, 32, 32, torch.float32, 64, seed=4)


def test_strong_decay(K):
    S0, p, cu = I.prefill_inputs([192], 2, 64, 64, dtype=torch.float32, seed=11, g_min=-10.0)
    o, S_fin, _, _, _ = run_prefill(K, S0, p, cu, 2, 64, 64, 0)
    args = [f(S0)] + [f(p[n]) for n in ("q", "k", "v", "g", "beta")]
    o_ref, S_ref, _ = O.prefill_recurrent(*args, cu_seqlens=cu, ckpt_stride=0)
    assert torch.isfinite(o).all() and torch.isfinite(S_fin).all()
    assert rel(o, o_ref) < TOL_F32 and rel(S_fin, S_ref) < TOL_F32


def test_resume_from_checkpoint_page(K):
    """Prefill 512 tokens, then resume the next 256 from the emitted page: equals 768 in one go."""
    H, d = 2, 64
    S0, p, cu = I.prefill_inputs([768], H, d, d, dtype=torch.float32, seed=12)
    o_all, S_all, pool, ids, _ = run_prefill(K, S0, p, cu, H, d, d, 512)
    resume = pool.page(int(ids[0]))[: H * d * d].reshape(1, H, d, d).clone()
    tail = {n: t[512:] for n, t in p.items()}
    o_tail, S_tail, _, _, _ = run_prefill(K, resume.cpu(), tail, [0, 256], H, d, d, 0)
    assert rel(S_tail, S_all) < TOL_F32
    assert rel(o_tail, o_all[512:]) < TOL_F32


@pytest.fixture
def chain_cols(K):
    yield K.kda_set_prefill_chain_columns
    K.kda_set_prefill_chain_columns(0)


def _np(t):
    return t.detach().to("cpu", torch.float32).numpy()


@pytest.fixture(scope="module")
def long_case():
    """B=1, H=32, dk=dv=128, T=8192, bf16, checkpoints every 512 tokens: the inputs on the
    device and the fp64 oracle of every head (one worker process per head)."""
    from oracle_pool import prefill_chunked_per_head
    H, d, T, stride = 32, 128, 8192, 512
    S0, p, cu = I.prefill_inputs([T], H, d, d, dtype=torch.bfloat16, seed=0, device="cuda")
    ref = prefill_chunked_per_head(_np(S0), *(_np(p[n]) for n in ("q", "k", "v", "g", "beta")), cu,
                                   stride, range(H))
    return S0, p, cu, ref


@pytest.mark.parametrize("cols", [0, 64])
def test_long_prefill_all_heads(K, cols, chain_cols, long_case):
    """B=1, H=32, dk=dv=128, T=8192, bf16, 16 checkpoints: outputs, final state and all 16
    checkpoint pages of every head against the fp64 oracle (chain CTA width chosen per call,
    which takes 32-column slices here, and forced to 64)."""
    chain_cols(cols)
    S0, p, cu, ref = long_case
    H, d, T, stride = 32, 128, 8192, 512
    n_ck = K.kda_num_checkpoints(cu, T, stride)
    assert n_ck == 16
    pool = K.PagePool(H * d * d * 4, n_ck)
    ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device="cuda")
    pos = torch.empty(n_ck, dtype=torch.int32, device="cuda")
    o, S_fin = K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                                     ckpt_stride=stride, page_pool=pool, ckpt_page_ids=ids,
                                     ckpt_pos=pos)
    torch.cuda.synchronize()
    assert K.kda_device_errors() == 0
    assert pos.tolist() == [512 * j for j in range(1, 17)]
    assert torch.equal(pool.page(int(ids[-1])).reshape(1, H, d, d), S_fin)
    pages = torch.stack([pool.page(int(ids[c])).reshape(H, d, d) for c in range(n_ck)])
    for h in range(H):
        o_ref, S_ref, ck_ref = ref[h]
        assert rel(o[:, h], o_ref[:, 0]) < TOL_BF16_OUT, h
        assert rel(S_fin[0, h], S_ref[0, 0]) < TOL_BF16_STATE, h
        assert [t for _, t, _ in ck_ref] == pos.tolist()
        for c in range(n_ck):
            assert rel(pages[c, h], ck_ref[c][2][0]) < TOL_BF16_STATE, (h, c)


def test_varlen_resume_longest_sequence_all_heads(K):
    """64 sequences, lengths log-uniform in [512, 32768] (multiples of 64), H=32, dk=dv=128, bf16,
    S0 ~ N(0, 0.05), checkpoints every 512 tokens: every head of the longest sequence (outputs,
    final state, every checkpoint page) and one head each of the shortest and the median."""
    from oracle_pool import prefill_chunked_per_head
    H, d, stride = 32, 128, 512
    lengths = I.varlen_lengths(64, seed=0)
    S0, p, cu = I.prefill_inputs(lengths, H, d, d, dtype=torch.bfloat16, seed=0, device="cuda")
    T = cu[-1]
    n_ck = K.kda_num_checkpoints(cu, T, stride)
    assert n_ck == sum(L // stride for L in lengths)
    pool = K.PagePool(H * d * d * 4, n_ck)
    ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device="cuda")
    pos = torch.empty(n_ck, dtype=torch.int32, device="cuda")
    o, S_fin = K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                                     ckpt_stride=stride, page_pool=pool, ckpt_page_ids=ids,
                                     ckpt_pos=pos)
    torch.cuda.synchronize()
    assert K.kda_device_errors() == 0
    expect = [t for L in lengths for t in O.checkpoint_positions(L, stride)]
    assert pos.tolist() == expect
    order = np.argsort(lengths)
    base = np.concatenate([[0], np.cumsum([L // stride for L in lengths])])

    def check(n, heads):
        a, b = cu[n], cu[n + 1]
        ins = [_np(S0[n:n + 1])] + [_np(p[x][a:b]) for x in ("q", "k", "v", "g", "beta")]
        ref = prefill_chunked_per_head(*ins, None, stride, heads)
        for h in heads:
            o_ref, S_ref, ck_ref = ref[h]
            assert rel(o[a:b, h], o_ref[:, 0]) < TOL_BF16_OUT, (n, h)
            assert rel(S_fin[n, h], S_ref[0, 0]) < TOL_BF16_STATE, (n, h)
            assert len(ck_ref) == lengths[n] // stride
            for j in range(len(ck_ref)):
                page = pool.page(int(ids[base[n] + j])).reshape(H, d, d)
                assert rel(page[h], ck_ref[j][2][0]) < TOL_BF16_STATE, (n, h, j)

    check(int(order[-1]), range(H))                       # the longest sequence, every head
    check(int(order[0]), [5])
    check(int(order[32]), [20])


# ---------------------------------------------------------------------------
# Tensor-core path (bf16, dk = 128, dv in {64, 128}) against the oracle
# ---------------------------------------------------------------------------
def _tc_case(K, lengths, dv, mode=0, seed=0, stride=128, g_min=-5.0, pad_bytes=0, state_std=0.05):
    H, dk = 2, 128
    S0, p, cu = I.prefill_inputs(lengths, H, dk, dv, dtype=torch.bfloat16, seed=seed,
                                 g_min=g_min, state_std=state_std)
    assert K.kda_prefill_workspace_bytes(cu, cu[-1], H, dk, dv, torch.bfloat16) > 0 or cu[-1] == 0
    o, S_fin, pool, ids, pos = run_prefill(K, S0, p, cu, H, dk, dv, stride, mode, pad_bytes)
    assert K.kda_device_errors() == 0
    args = [f(S0)] + [f(p[n]) for n in ("q", "k", "v", "g", "beta")]
    o_ref, S_ref, ck_ref = O.prefill_chunked(*args, cu_seqlens=cu, chunk=64, ckpt_stride=stride,
                                             mode=mode)
    assert rel(o, o_ref) < TOL_BF16_OUT
    assert rel(S_fin, S_ref) < TOL_BF16_STATE
    assert pos.tolist() == [t for _, t, _ in ck_ref]
    n_state = H * dk * dv
    for c, (n, t, st) in enumerate(ck_ref):
        page = pool.page(int(ids[c]))
        assert rel(page[:n_state].reshape(H, dk, dv), st) < TOL_BF16_STATE
        if pad_bytes:
            assert torch.all(page[n_state:] == 0)
        if t == lengths[n]:
            assert torch.equal(page[:n_state].reshape(H, dk, dv), S_fin[n])
    return o, S_fin, o_ref, S_ref


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dv", [64, 128])
def test_tc_single_sequence(K, dv, mode):
    _tc_case(K, [512], dv, mode=mode, seed=dv + mode)


@pytest.mark.parametrize("dv", [64, 128])
def test_tc_ragged_varlen(K, dv):
    _tc_case(K, [1, 63, 65, 130, 0, 200, 128, 320], dv, seed=3, pad_bytes=64)


def test_tc_strong_decay(K):
    _tc_case(K, [256, 100], 128, seed=4, g_min=-10.0)


@pytest.mark.parametrize("mode", [0, 1])
def test_tc_weak_decay_long_memory(K, mode):
    """g = -0.01 sigmoid(.): the state keeps nearly all of its past over 2048 tokens (32
    chunks), so the bf16 operand copies of S feed 32 chained updates; outputs, final state
    and every checkpoint page must still meet the bf16 tolerances."""
    _tc_case(K, [2048], 128, mode=mode, seed=9, stride=512, g_min=-0.01)


@pytest.mark.parametrize("cols", [32, 64])
@pytest.mark.parametrize("dv", [64, 128])
def test_tc_chain_column_slices(K, dv, cols, chain_cols):
    """Both chain CTA widths, forced, on ragged sequences in both modes."""
    chain_cols(cols)
    _tc_case(K, [1, 63, 65, 130, 0, 200, 128, 320], dv, mode=0, seed=11, pad_bytes=64)
    _tc_case(K, [300, 64], dv, mode=1, seed=12, stride=64)


def test_tc_chain_widths_agree(K, chain_cols):
    """32- and 64-column chain CTAs compute every state column the same way."""
    H, d = 4, 128
    S0, p, cu = I.prefill_inputs([900, 77, 256], H, d, d, dtype=torch.bfloat16, seed=13, device="cuda")
    res = []
    for cols in (32, 64):
        chain_cols(cols)
        res.append(K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                                         ckpt_stride=0))
    torch.cuda.synchronize()
    assert K.kda_device_errors() == 0
    (o32, s32), (o64, s64) = res
    assert rel(o32, o64) < 1e-5 and rel(s32, s64) < 1e-5


def test_tc_cold_start_and_single_chunk(K):
    _tc_case(K, [64], 128, seed=5, state_std=0.0)
    _tc_case(K, [7], 64, seed=6)


def test_tc_matches_fp32_kernel(K):
    """bf16 inputs: tensor-core kernels vs the fp32 CUDA-core kernel on the same call."""
    H, d = 4, 128
    S0, p, cu = I.prefill_inputs([700, 300], H, d, d, dtype=torch.bfloat16, seed=8, device="cuda")
    o_tc, S_tc = K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                                       ckpt_stride=0)
    o_ref, S_ref = K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                                         ckpt_stride=0, workspace=None)
    torch.cuda.synchronize()
    assert rel(o_tc, o_ref) < TOL_BF16_OUT and rel(S_tc, S_ref) < TOL_BF16_STATE


def test_tc_workspace_too_small_is_rejected(K):
    H, d = 2, 128
    S0, p, cu = I.prefill_inputs([128], H, d, d, dtype=torch.bfloat16, seed=1, device="cuda")
    need = K.kda_prefill_workspace_bytes(cu, 128, H, d, d, torch.bfloat16)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(K.KdaError) as e:
        K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                              ckpt_stride=0, workspace=ws)
    assert e.value.status == -2


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 64)])
def test_gate_outside_contract_is_flagged(K, dtype, dk, dv):
    """The chunked kernels take g in [-10, 0] ([SERVE] §1.3 draws g = g_min sigmoid(.) in
    [g_min, 0]; the block-reference factors reach e^(8 |g|)).  Gates drawn with g_min = -20
    (about half of them below -10), or one NaN gate, raise DEVERR_GATE; gates drawn with
    g_min = -10 raise nothing.  Both the tensor-core (bf16, dk = 128) and the CUDA-core
    kernels are checked."""
    H = 2
    K.kda_device_errors()                                    # start from a clear word

    def run(g_min, nan=False):
        S0, p, cu = I.prefill_inputs([192], H, dk, dv, dtype=dtype, seed=5, g_min=g_min, device="cuda")
        if nan:
            p["g"][100, 1, 7] = float("nan")
        K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu, ckpt_stride=0)
        torch.cuda.synchronize()
        return p, K.kda_device_errors()

    p, flags = run(-10.0)
    assert float(p["g"].min()) >= -10.0 and flags == 0
    p, flags = run(-20.0)
    assert bool((p["g"] < -10).any()) and flags & K.DEVERR_GATE
    _, flags = run(-5.0, nan=True)
    assert flags & K.DEVERR_GATE
