"""GPU parity of the slot-pool entry points (kda_decode_step_slots, kda_verify_replay_slots):
states kept in a [layers, slots, H, ...] pool in either layout, (dk, dv) or transposed (dv, dk),
against the fp64 oracle run on the gathered (and, for the transposed layout, transposed back)
states.  Slots no row names, and rows whose slot id is out of range, must stay untouched."""
import numpy as np
import pytest
import torch

from kda_delta_rule_gb300 import inputs as I
from oracle import kda_oracle as O
from parity import TOL_BF16_STORED_OUT, TOL_F32, rel

pytestmark = pytest.mark.gpu
f = I.to_f64_numpy
DIMS = [(dk, dv) for dk in (32, 64, 128) for dv in (32, 64, 128)]


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


def _to_layout(S, layout, K):
    """(…, dk, dv) states -> the pool's stored form."""
    return S.transpose(-1, -2).contiguous() if layout == K.LAYOUT_VK else S.contiguous()


def _from_layout(P, layout, K):
    return P.transpose(-1, -2) if layout == K.LAYOUT_VK else P


def _pool(n_slots, lead, H, dk, dv, seed):
    gen = torch.Generator().manual_seed(seed)
    return 0.1 * torch.randn(*lead, n_slots, H, dk, dv, generator=gen, dtype=torch.float64)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", DIMS)
def test_decode_slots_transposed(K, dk, dv, dtype, mode):
    B, H, n_slots = 5, 4, 11
    _, p = I.decode_inputs(B, H, dk, dv, dtype=dtype, seed=7 * dk + dv + mode)
    S_math = _pool(n_slots, (), H, dk, dv, seed=dk * dv + mode)          # (slots, H, dk, dv) f64
    slots = torch.tensor([9, 2, -1, 0, 6], dtype=torch.int32)             # row 2 is padding
    pool = _to_layout(S_math.float(), K.LAYOUT_VK, K).cuda()
    before = pool.clone()
    pd = {n: t.cuda() for n, t in p.items()}
    o = K.kda_decode_step_slots(pool, slots.cuda(), pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"],
                                layout=K.LAYOUT_VK, mode=mode)
    live = [b for b in range(B) if slots[b] >= 0]
    S0 = np.stack([f(S_math[int(slots[b])].float()) for b in live])
    o_ref, S_ref = O.kda_step(S0, *(f(p[n][live]) for n in ("q", "k", "v", "g", "beta")), mode)
    torch.cuda.synchronize()
    got_S = torch.stack([_from_layout(pool[int(slots[b])], K.LAYOUT_VK, K) for b in live])
    assert rel(got_S, S_ref) < TOL_F32
    assert rel(o[live], o_ref) < (TOL_F32 if dtype == torch.float32 else TOL_BF16_STORED_OUT)
    assert torch.count_nonzero(o[2]) == 0
    untouched = [s for s in range(n_slots) if s not in [int(slots[b]) for b in live]]
    assert torch.equal(pool[untouched], before[untouched])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(32, 64), (128, 128), (64, 32)])
def test_decode_slots_kv_matches_dense_call(K, dk, dv, dtype):
    """Layout (dk, dv) through a pool gives the bits of kda_decode_step on the gathered states."""
    B, H, n_slots = 6, 4, 9
    _, p = I.decode_inputs(B, H, dk, dv, dtype=dtype, seed=3)
    pool = _pool(n_slots, (), H, dk, dv, seed=4).float().cuda()
    slots = torch.tensor([4, 0, 8, 3, 1, 7], dtype=torch.int32, device="cuda")
    dense = pool[slots.long()].clone()
    pd = {n: t.cuda() for n, t in p.items()}
    o_dense = K.kda_decode_step(dense, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"])
    o_slots = K.kda_decode_step_slots(pool, slots, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"],
                                      layout=K.LAYOUT_KV)
    torch.cuda.synchronize()
    assert torch.equal(o_slots, o_dense)
    assert torch.equal(pool[slots.long()], dense)


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
def test_replay_slots_ping_pong(K, dk, dv, dtype, layout):
    """Three layers, committed states read from one set of slots and the replayed states
    written to another set of the same pool; accepted counts 0 .. draft; one padded row."""
    Lr, B, H, draft, n_slots = 3, 5, 2, 6, 12
    _, proj, _ = I.replay_inputs(B, H, dk, dv, draft, dtype=dtype, seed=dk + dv + layout)
    # per-layer projections: the first layer's draw, then fresh draws for the others
    P = {n: [getattr(proj, n)] for n in ("q", "k", "v", "g", "beta")}
    for layer in range(1, Lr):
        _, pl, _ = I.replay_inputs(B, H, dk, dv, draft, dtype=dtype, seed=100 * layer + dk + dv)
        for n in P:
            P[n].append(getattr(pl, n))
    P = {n: torch.stack(v).contiguous() for n, v in P.items()}          # (L, draft, B, H, D)
    n_acc = torch.tensor([draft, 0, 3, 1, 5], dtype=torch.int32)
    slot_in = torch.tensor([1, 5, 7, -1, 10], dtype=torch.int32)
    slot_out = torch.tensor([0, 2, 11, 4, 3], dtype=torch.int32)
    S_math = _pool(n_slots, (Lr,), H, dk, dv, seed=dk * 3 + dv)
    pool = _to_layout(S_math.float(), layout, K).cuda()
    before = pool.clone()
    pd = {n: t.cuda() for n, t in P.items()}
    _, out = K.kda_verify_replay_slots(pool, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"], n_acc.cuda(),
                                       slot_in.cuda(), slot_out.cuda(), S_pool_new=pool, layout=layout)
    torch.cuda.synchronize()
    live = [b for b in range(B) if slot_in[b] >= 0]
    tol_o = TOL_F32 if dtype == torch.float32 else TOL_BF16_STORED_OUT
    for layer in range(Lr):
        S0 = np.stack([f(S_math[layer, int(slot_in[b])].float()) for b in live])
        S_ref, out_ref = O.verify_and_replay_batched(
            S0, *(f(P[n][layer][:, live]) for n in ("q", "k", "v", "g", "beta")), n_acc[live].numpy())
        got = torch.stack([_from_layout(pool[layer, int(slot_out[b])], layout, K) for b in live])
        assert rel(got, S_ref) < TOL_F32
        assert rel(out[layer][live], out_ref) < tol_o
        assert torch.count_nonzero(out[layer][3]) == 0                   # padded row
        for b in live:
            assert torch.count_nonzero(out[layer][b][:, int(n_acc[b]):]) == 0
    written = {int(slot_out[b]) for b in live}
    kept = [s for s in range(n_slots) if s not in written]
    assert torch.equal(pool[:, kept], before[:, kept])                   # committed + unnamed slots


def test_replay_slots_kv_matches_layers_call(K):
    """Layout (dk, dv), separate output pool: same bits as kda_verify_replay_layers."""
    Lr, B, H, dk, dv, draft, n_slots = 2, 4, 3, 64, 64, 5, 7
    P = {n: [] for n in ("q", "k", "v", "g", "beta")}
    for layer in range(Lr):
        _, pl, _ = I.replay_inputs(B, H, dk, dv, draft, dtype=torch.bfloat16, seed=40 + layer)
        for n in P:
            P[n].append(getattr(pl, n))
    pd = {n: torch.stack(v).contiguous().cuda() for n, v in P.items()}
    n_acc = torch.tensor([5, 2, 0, 4], dtype=torch.int32, device="cuda")
    slots = torch.tensor([6, 1, 3, 0], dtype=torch.int32, device="cuda")
    pool = _pool(n_slots, (Lr,), H, dk, dv, seed=41).float().cuda()
    dense = pool[:, slots.long()].contiguous()
    S_dense, out_dense = K.kda_verify_replay_layers(dense, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"],
                                                    n_acc)
    new_pool, out = K.kda_verify_replay_slots(pool, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"], n_acc,
                                              slots, layout=K.LAYOUT_KV)
    torch.cuda.synchronize()
    assert torch.equal(out, out_dense)
    assert torch.equal(new_pool[:, slots.long()], S_dense)


def test_decode_slots_transposed_full_size_sampled(K):
    """B=256, H=32, dk=dv=128, bf16, pool of 512 transposed slots; 4 steps, 6 heads checked."""
    B, H, d, n_slots, steps = 256, 32, 128, 512, 4
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1)
    pool = (0.05 * torch.randn(n_slots, H, d, d, generator=gen, device="cuda")).contiguous()
    slots = torch.randperm(n_slots, generator=gen, device="cuda")[:B].to(torch.int32)
    sample = [(0, 0), (17, 5), (100, 31), (255, 12), (128, 16), (3, 30)]
    S_ref = np.stack([f(pool[int(slots[b]), h].T) for b, h in sample])
    o = torch.empty(B, H, d, device="cuda", dtype=torch.bfloat16)
    for t in range(steps):
        p = I.decode_step_projections(B, H, d, d, dtype=torch.bfloat16, seed=500 + t, device="cuda")
        K.kda_decode_step_slots(pool, slots, p["q"], p["k"], p["v"], p["g"], p["beta"], o=o,
                                layout=K.LAYOUT_VK)
        cols = {n: np.stack([f(p[n][b, h]) for b, h in sample]) for n in ("q", "k", "v", "g", "beta")}
        o_ref, S_ref = O.kda_step(S_ref, cols["q"], cols["k"], cols["v"], cols["g"], cols["beta"])
        got = torch.stack([o[b, h] for b, h in sample])
        assert rel(got, o_ref) < TOL_BF16_STORED_OUT
    torch.cuda.synchronize()
    got_S = torch.stack([pool[int(slots[b]), h].T for b, h in sample])
    assert rel(got_S, S_ref) < TOL_F32
