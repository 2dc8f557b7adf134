"""pack_heads / unpack_heads and store_kda / load_kda on the GPU: bit-exact."""
import pytest
import torch

from oracle import kda_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


@pytest.mark.parametrize("B,H,dk,dv", [(1, 32, 128, 128), (3, 5, 32, 64), (2, 1, 64, 32)])
def test_pack_matches_oracle_layout_and_roundtrips(K, B, H, dk, dv):
    S = torch.randn(B, H, dk, dv, device="cuda")
    flat = K.kda_pack_heads(S, flat_elems=S.numel() + 37)
    ref = O.pack_heads(S.cpu().numpy())
    torch.cuda.synchronize()
    assert torch.equal(flat[: S.numel()].cpu(), torch.from_numpy(ref))
    assert torch.all(flat[S.numel():] == 0)
    back = K.kda_unpack_heads(flat, torch.empty_like(S))
    torch.cuda.synchronize()
    assert torch.equal(back, S)


def test_pack_strided_slot_of_a_batched_state(K):
    big = torch.randn(6, 4, 64, 64, device="cuda")
    sl = big[2:5, 1:3]                       # (3, 2, 64, 64), strided over b and h
    flat = K.kda_pack_heads(sl)
    torch.cuda.synchronize()
    assert torch.equal(flat, sl.contiguous().reshape(-1))
    out = torch.zeros_like(big)
    K.kda_unpack_heads(flat, out[2:5, 1:3])
    torch.cuda.synchronize()
    assert torch.equal(out[2:5, 1:3], sl) and torch.all(out[:2] == 0)


def test_store_load_kda_pages(K):
    B, H, d = 2, 4, 32
    pool = K.PagePool(B * H * d * d * 4 + 256, 4)
    pool.arena.fill_(0x7F)
    ids = pool.alloc(2, K.PAGE_KDA_STATE)
    mla = pool.alloc(1, K.PAGE_MLA_KV)
    S = torch.randn(B, H, d, d, device="cuda")
    pool.store_kda(ids[1], S)
    got = pool.load_kda(ids[1], torch.empty_like(S))
    torch.cuda.synchronize()
    assert torch.equal(got, S)
    page = pool.page(ids[1])
    assert torch.all(page[S.numel():] == 0)
    with pytest.raises(K.KdaError):
        pool.store_kda(mla[0], S)
    pool.free(ids + mla)
    assert pool.num_free() == 4
