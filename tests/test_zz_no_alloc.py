"""The allocation-free prefill entry point, kda_prefill_chunked_noalloc, on the GPU.

Some callers cannot allocate device memory when they call the prefill: a
serving loop that forbids cudaMalloc/cudaFree on its hot path (they
synchronise the whole device and stall every stream), or code running inside a
framework that owns all device memory through its own allocator.  For them the
library takes the tensor-core scratch from one fixed device array that it
carries itself.  These tests call that entry point through the C ABI and check,
on two calls in a row, that outputs, final states and checkpoint pages match
the regular entry point given a caller workspace; and that a call needing more
scratch than the array holds is refused without running.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

from kda_delta_rule_gb300 import inputs as I
from parity import TOL_BF16_OUT, TOL_BF16_STATE, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc_call(K, S0, p, cu, H, dk, dv, stride, pool, ids, pos, o, S_fin, dtype=None):
    T = cu[-1]
    arr = (ctypes.c_int32 * len(cu))(*cu)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return K._lib.kda_prefill_chunked_noalloc(
        _ptr(S0), _ptr(p["q"]), _ptr(p["k"]), _ptr(p["v"]), _ptr(p["g"]), _ptr(p["beta"]),
        arr, len(cu) - 1, T, H, dk, dv, K.KDA_BF16 if dtype is None else dtype, 64, stride, _ptr(o),
        _ptr(S_fin), ctypes.c_void_p(pool.arena.data_ptr()), pool.page_bytes, _ptr(ids), _ptr(pos),
        ids.numel(), K.DECAY_FIRST, stream)


def _one_call(K, lengths, seed, H=4, dk=128, dv=128, dtype=torch.bfloat16, stride=128):
    S0, p, cu = I.prefill_inputs(lengths, H, dk, dv, dtype=dtype, seed=seed, device="cuda")
    T = cu[-1]
    need = K.kda_prefill_workspace_bytes(cu, T, H, dk, dv, dtype)
    assert need <= (64 << 20)                     # fits the built-in scratch (0: CUDA-core kernel)
    n_ck = K.kda_num_checkpoints(cu, T, stride)
    page_bytes = H * dk * dv * 4 + 256
    pools, outs = [], []
    for _ in range(2):
        pool = K.PagePool(page_bytes, n_ck)
        pool.arena.fill_(0x5A)
        ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device="cuda")
        pos = torch.full((n_ck,), -1, dtype=torch.int32, device="cuda")
        o = torch.empty(T, H, dv, dtype=dtype, device="cuda")
        S_fin = torch.empty_like(S0)
        pools.append((pool, ids, pos))
        outs.append((o, S_fin))
    # regular entry point: with a caller workspace where the shape takes one, else without
    pool, ids, pos = pools[0]
    K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                          ckpt_stride=stride, page_pool=pool, ckpt_page_ids=ids, ckpt_pos=pos,
                          o=outs[0][0], S_final=outs[0][1], workspace="auto" if need > 0 else None)
    # allocation-free entry point, straight through the C ABI
    pool, ids, pos = pools[1]
    code = K.KDA_BF16 if dtype == torch.bfloat16 else K.KDA_F32
    st = _noalloc_call(K, S0, p, cu, H, dk, dv, stride, pool, ids, pos, *outs[1], dtype=code)
    assert st == 0, K._lib.kda_last_error()
    torch.cuda.synchronize()
    assert K.kda_device_errors() == 0
    (o_ref, S_ref), (o_na, S_na) = outs
    # both calls run the same kernels on the same inputs: the results agree bit for bit
    # (a stale or partly overwritten scratch would show here); the tolerances only
    # describe the size of a difference if there is one
    assert torch.equal(o_na, o_ref), f"outputs differ, rel {rel(o_na, o_ref):.3g} (bf16 bound {TOL_BF16_OUT})"
    assert torch.equal(S_na, S_ref), f"final states differ, rel {rel(S_na, S_ref):.3g} (bound {TOL_BF16_STATE})"
    assert torch.equal(pools[1][2], pools[0][2])                 # checkpoint positions
    n_state = H * dk * dv
    for c in range(n_ck):
        a = pools[0][0].page(int(pools[0][1][c]))
        b = pools[1][0].page(int(pools[1][1][c]))
        assert torch.equal(b[:n_state], a[:n_state]), f"checkpoint {c} differs"
        assert torch.all(b[n_state:] == 0)
    return need


def test_noalloc_matches_workspace_entry_point_twice(K):
    # two calls in a row: the second reuses the scratch the first one left behind
    assert _one_call(K, [200, 64, 130], seed=21) > 0
    assert _one_call(K, [320, 5, 0, 257], seed=22) > 0


def test_noalloc_without_scratch_runs_the_cuda_core_kernel(K):
    # fp32 projections and a dk other than 128 need no scratch: the call runs the fp32
    # CUDA-core kernel, exactly as kda_prefill_chunked does with a NULL workspace
    assert _one_call(K, [130, 64], seed=23, H=2, dk=64, dv=64, dtype=torch.float32, stride=64) == 0
    assert _one_call(K, [100], seed=24, H=2, dk=32, dv=128, dtype=torch.bfloat16, stride=64) == 0


def test_noalloc_refuses_calls_larger_than_its_scratch(K):
    H, d, T = 32, 128, 2048          # 32 chunks x 32 heads of scratch: more than the array holds
    S0, p, cu = I.prefill_inputs([T], H, d, d, dtype=torch.bfloat16, seed=3, device="cuda")
    need = K.kda_prefill_workspace_bytes(cu, T, H, d, d, torch.bfloat16)
    assert need > (64 << 20)
    pool = K.PagePool(H * d * d * 4, 4)
    ids = torch.tensor(pool.alloc(4), dtype=torch.int32, device="cuda")
    pos = torch.zeros(4, dtype=torch.int32, device="cuda")
    o = torch.zeros(T, H, d, dtype=torch.bfloat16, device="cuda")
    S_fin = torch.zeros_like(S0)
    st = _noalloc_call(K, S0, p, cu, H, d, d, 512, pool, ids, pos, o, S_fin)
    assert st == -2
    assert b"scratch" in K._lib.kda_last_error()
    torch.cuda.synchronize()
    assert torch.all(S_fin == 0) and torch.all(o == 0)           # nothing ran
