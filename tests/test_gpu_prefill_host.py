"""Prefill from host memory (kda_prefill_chunked_host): the segmented, copy-overlapped call
gives the same bits as the device-resident call, including checkpoint pages and positions."""
import pytest
import torch

from kda_delta_rule_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


def _both(K, lengths, H, dk, dv, dtype, stride, segment, mode=0, seed=0, S0_none=False):
    S0, p, cu = I.prefill_inputs(lengths, H, dk, dv, dtype=dtype, seed=seed)
    T = cu[-1]
    N = len(lengths)
    n_ck = K.kda_num_checkpoints(cu, T, stride)
    page_bytes = H * dk * dv * 4
    ref_pool = K.PagePool(page_bytes, max(n_ck, 1))
    host_pool = K.PagePool(page_bytes, max(n_ck, 1))
    ids = torch.arange(n_ck, dtype=torch.int32, device="cuda").flip(0).contiguous()
    ref_pos = torch.full((max(n_ck, 1),), -1, dtype=torch.int32, device="cuda")[:n_ck]
    host_pos = torch.full((max(n_ck, 1),), -1, dtype=torch.int32, device="cuda")[:n_ck]
    host_pool.arena.fill_(0xAB)
    if n_ck:
        ref_pool.alloc(n_ck)
        host_pool.alloc(n_ck)
    pd = {n: t.cuda() for n, t in p.items()}
    o_ref, S_ref = K.kda_prefill_chunked(None if S0_none else S0.cuda(), pd["q"], pd["k"], pd["v"], pd["g"],
                                         pd["beta"], cu_seqlens=cu, ckpt_stride=stride, page_pool=ref_pool,
                                         ckpt_page_ids=ids if n_ck else None, ckpt_pos=ref_pos if n_ck else None,
                                         mode=mode)
    ph = {n: t.contiguous().pin_memory() for n, t in p.items()}
    S0h = None if S0_none else S0.contiguous().pin_memory()
    o_h = torch.empty((T, H, dv), dtype=dtype).pin_memory()
    S_h = torch.empty((N, H, dk, dv), dtype=torch.float32).pin_memory()
    scratch = torch.empty(K.kda_prefill_host_scratch_bytes(H, dk, dv, dtype, stride, segment),
                          dtype=torch.uint8, device="cuda")
    K.kda_prefill_chunked_host(S0h, ph["q"], ph["k"], ph["v"], ph["g"], ph["beta"], o_h, S_h, scratch,
                               cu_seqlens=cu, ckpt_stride=stride, page_pool=host_pool,
                               ckpt_page_ids=ids if n_ck else None, ckpt_pos=host_pos if n_ck else None,
                               segment_tokens=segment, mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_ref.cpu())
    assert torch.equal(S_h, S_ref.cpu())
    if n_ck:
        assert torch.equal(host_pool.arena, ref_pool.arena)
        assert torch.equal(host_pos, ref_pos)
    return n_ck


def test_host_single_sequence_cut_at_checkpoints(K):
    """T=1536 in 512-token segments: two cuts, each at a checkpoint; bf16 tensor-core path."""
    assert _both(K, [1536], 2, 128, 128, torch.bfloat16, 512, 512) == 3


def test_host_varlen_pieces_and_empty_sequence(K):
    """Several sequences, one split across segments, one empty, undecayed-delta mode."""
    assert _both(K, [700, 64, 0, 1300, 129], 2, 128, 64, torch.bfloat16, 128, 256, mode=1, seed=3) > 0


def test_host_fp32_cuda_core_path_zero_state(K):
    _both(K, [300, 900], 3, 64, 64, torch.float32, 0, 320, seed=5, S0_none=True)


def test_host_more_pieces_than_a_segment_holds(K):
    """Twelve short sequences: segments close at eight pieces."""
    _both(K, [64] * 12, 2, 32, 32, torch.float32, 64, 4096, seed=7)
