"""GPU parity of the decode step and verify/replay kernels against the fp64 oracle."""
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


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", DIMS)
def test_decode_step(K, dk, dv, dtype, mode):
    B, H = 3, 4
    S, p = I.decode_inputs(B, H, dk, dv, dtype=dtype, seed=dk + dv + mode, state_std=0.1)
    Sd = S.cuda()
    pd = {n: t.cuda() for n, t in p.items()}
    o = K.kda_decode_step(Sd, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"], mode=mode)
    o_ref, S_ref = O.kda_step(f(S), f(p["q"]), f(p["k"]), f(p["v"]), f(p["g"]), f(p["beta"]), mode)
    torch.cuda.synchronize()
    assert rel(Sd, S_ref) < TOL_F32
    assert rel(o, o_ref) < (TOL_F32 if dtype == torch.float32 else TOL_BF16_STORED_OUT)


@pytest.mark.parametrize("H", [1, 3, 5])
def test_decode_odd_head_counts(K, H):
    S, p = I.decode_inputs(7, H, 32, 32, dtype=torch.float32, seed=H)
    Sd = S.cuda()
    pd = {n: t.cuda() for n, t in p.items()}
    o = K.kda_decode_step(Sd, pd["q"], pd["k"], pd["v"], pd["g"], pd["beta"])
    o_ref, S_ref = O.kda_step(f(S), f(p["q"]), f(p["k"]), f(p["v"]), f(p["g"]), f(p["beta"]))
    torch.cuda.synchronize()
    assert rel(Sd, S_ref) < TOL_F32 and rel(o, o_ref) < TOL_F32


def test_decode_batched_256_steps_sampled(K):
    """B=256, H=32, dk=dv=128, 256 steps with fresh bf16 projections; 6 heads checked."""
    B, H, d, steps = 256, 32, 128, 256
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    S = (0.05 * torch.randn(B, H, d, d, generator=gen, device="cuda")).contiguous()
    sample = [(0, 0), (17, 5), (100, 31), (255, 12), (128, 16), (3, 30)]
    S_ref = np.stack([f(S[b, h]) for b, h in sample])
    o = torch.empty(B, H, d, device="cuda", dtype=torch.bfloat16)
    for t in range(steps):
        p = I.decode_step_projections(B, H, d, d, dtype=torch.bfloat16, seed=1000 + t, device="cuda")
        K.kda_decode_step(S, p["q"], p["k"], p["v"], p["g"], p["beta"], o=o)
        cols = {n: np.stack([f(p[n][b, h]) for b, h in sample]) for n in ("q", "k", "v", "g", "beta")}
        o_ref, S_ref = O.kda_step(S_ref, cols["q"], cols["k"], cols["v"], cols["g"], cols["beta"])
        if t in (0, steps - 1):
            got = torch.stack([o[b, h] for b, h in sample])
            assert rel(got, o_ref) < TOL_BF16_STORED_OUT
    torch.cuda.synchronize()
    got_S = torch.stack([S[b, h] for b, h in sample])
    assert rel(got_S, S_ref) < TOL_F32


# ---------------------------------------------------------------------------
def _replay(K, B, H, dk, dv, draft, dtype, seed, mode=0, n_accepted=None, state_std=0.1):
    S, proj, n_acc = I.replay_inputs(B, H, dk, dv, draft, dtype=dtype, seed=seed,
                                     n_accepted=n_accepted, state_std=state_std)
    Sc = S.cuda()
    snapshot = Sc.clone()
    pr = proj.to("cuda")
    S_new, out = K.kda_verify_replay(Sc, pr.q, pr.k, pr.v, pr.g, pr.beta, n_acc.cuda(), mode=mode)
    S_ref, out_ref = O.verify_and_replay_batched(f(S), f(proj.q), f(proj.k), f(proj.v), f(proj.g),
                                                 f(proj.beta), n_acc.numpy(), mode)
    torch.cuda.synchronize()
    assert torch.equal(Sc, snapshot), "the committed state was written"
    return S_new, out, S_ref, out_ref, n_acc


@pytest.mark.parametrize("mode", [0, 1])
def test_replay_speculative_shape(K, mode):
    """B=32, H=16, dk=dv=32, draft 8, fp32, n_accepted ~ U{0..8}: whole batch checked."""
    S_new, out, S_ref, out_ref, n_acc = _replay(K, 32, 16, 32, 32, 8, torch.float32, 0, mode)
    assert rel(S_new, S_ref) < TOL_F32
    assert rel(out, out_ref) < TOL_F32
    for b, n in enumerate(n_acc.tolist()):
        assert torch.all(out[b, :, n:] == 0)


def test_replay_pages_three_scenarios(K):
    """Draft 4 with n = 2, 4, 0 (partial, all, none)."""
    S_new, out, S_ref, out_ref, _ = _replay(K, 3, 2, 32, 32, 4, torch.float32, 5,
                                            n_accepted=[2, 4, 0])
    assert rel(S_new, S_ref) < TOL_F32 and rel(out, out_ref) < TOL_F32


def test_replay_reject_all_is_identity(K):
    S, proj, _ = I.replay_inputs(4, 8, 64, 64, 6, dtype=torch.float32, seed=3)
    Sc = S.cuda()
    pr = proj.to("cuda")
    S_new, out = K.kda_verify_replay(Sc, pr.q, pr.k, pr.v, pr.g, pr.beta,
                                     torch.zeros(4, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(S_new, Sc) and torch.all(out == 0)


def test_replay_clamps_counts(K):
    S_new, out, S_ref, out_ref, _ = _replay(K, 4, 2, 32, 64, 3, torch.float32, 9,
                                            n_accepted=[-2, 9, 3, 1])
    # oracle clamps the same way
    assert rel(S_new, S_ref) < TOL_F32 and rel(out, out_ref) < TOL_F32


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32), (32, 128)])
def test_replay_bf16(K, dk, dv):
    S_new, out, S_ref, out_ref, _ = _replay(K, 5, 4, dk, dv, 8, torch.bfloat16, dk + dv)
    assert rel(S_new, S_ref) < TOL_F32 and rel(out, out_ref) < TOL_BF16_STORED_OUT


def test_replay_refuses_in_place(K):
    S, proj, n = I.replay_inputs(2, 2, 32, 32, 2, dtype=torch.float32, seed=1)
    Sc = S.cuda()
    pr = proj.to("cuda")
    with pytest.raises(K.KdaError) as e:
        K.kda_verify_replay(Sc, pr.q, pr.k, pr.v, pr.g, pr.beta, n.cuda(), S_new=Sc)
    assert e.value.status == -7


@pytest.mark.parametrize("trans", [False, True])
def test_small_head_replay_forms_agree(K, trans):
    """32 x 32 heads run one warp per head when the heads fill the GPU and two warps per
    head (16 columns each) when they would not: 4,096 stacked heads take the first form,
    each 512-head layer alone the second.  The two agree to fp32 rounding (their sums
    associate differently) and each stays within tolerance of the oracle; a transposed
    slot pool gives the same bits as the (dk, dv) states in either form."""
    Lr, B, H, D, draft = 8, 32, 16, 32, 8
    sets = [I.replay_inputs(B, H, D, D, draft, dtype=torch.float32, seed=90 + l) for l in range(Lr)]
    n_acc = sets[0][2].cuda()
    S = torch.stack([s_[0] for s_ in sets]).cuda()
    cat = lambda name: torch.stack([getattr(s_[1], name) for s_ in sets]).cuda()
    q, k, v, g, beta = (cat(nm) for nm in ("q", "k", "v", "g", "beta"))
    S_new, out = K.kda_verify_replay_layers(S, q, k, v, g, beta, n_acc)
    torch.cuda.synchronize()
    singles = []
    for l in range(Lr):
        S1, o1 = K.kda_verify_replay(S[l], q[l], k[l], v[l], g[l], beta[l], n_acc)
        torch.cuda.synchronize()
        singles.append((S1, o1))
        assert rel(S1, S_new[l]) < 1e-5 and rel(o1, out[l]) < 1e-5, f"layer {l}"
    for l in (0, Lr - 1):
        S_ref, out_ref = O.verify_and_replay_batched(f(S[l]), f(q[l]), f(k[l]), f(v[l]), f(g[l]), f(beta[l]),
                                                     n_acc.cpu().numpy())
        assert rel(S_new[l], S_ref) < TOL_F32 and rel(out[l], out_ref) < TOL_F32
        assert rel(singles[l][0], S_ref) < TOL_F32 and rel(singles[l][1], out_ref) < TOL_F32
    if trans:
        # the same layers from transposed pools of B slots each (identity slot ids):
        # the stacked call, then layer 0 alone (the other form)
        pool = S.transpose(-1, -2).contiguous()
        ids = torch.arange(B, dtype=torch.int32, device="cuda")
        pool_new, o_t = K.kda_verify_replay_slots(pool, q, k, v, g, beta, n_acc, ids, layout=K.LAYOUT_VK)
        p0_new, o0 = K.kda_verify_replay_slots(pool[:1], q[:1], k[:1], v[:1], g[:1], beta[:1], n_acc, ids,
                                               layout=K.LAYOUT_VK)
        torch.cuda.synchronize()
        assert torch.equal(o_t, out) and torch.equal(pool_new.transpose(-1, -2), S_new)
        assert torch.equal(o0[0], singles[0][1]) and torch.equal(p0_new[0].transpose(-1, -2), singles[0][0])


@pytest.mark.parametrize("dk,dv,dtype", [(32, 32, torch.float32), (128, 128, torch.bfloat16)])
def test_replay_layers_match_single_calls_and_oracle(K, dk, dv, dtype):
    """Three stacked layers in one launch: bit-identical to three single-layer calls,
    each layer within tolerance of the oracle, committed states untouched."""
    Lr, B, H, draft = 3, 4, 4, 6
    sets = [I.replay_inputs(B, H, dk, dv, draft, dtype=dtype, seed=40 + l) for l in range(Lr)]
    n_acc = sets[0][2].cuda()                      # the accepted count is per sequence, shared
    S = torch.stack([s[0] for s in sets]).cuda()
    cat = lambda name: torch.stack([getattr(s[1], name) for s in sets]).cuda()
    q, k, v, g, beta = (cat(n) for n in ("q", "k", "v", "g", "beta"))
    snapshot = S.clone()
    S_new, out = K.kda_verify_replay_layers(S, q, k, v, g, beta, n_acc)
    torch.cuda.synchronize()
    assert torch.equal(S, snapshot), "a committed state was written"
    tol_out = TOL_F32 if dtype == torch.float32 else TOL_BF16_STORED_OUT
    for l in range(Lr):
        S1, o1 = K.kda_verify_replay(S[l], q[l], k[l], v[l], g[l], beta[l], n_acc)
        torch.cuda.synchronize()
        assert torch.equal(S1, S_new[l]) and torch.equal(o1, out[l])
        S_ref, out_ref = O.verify_and_replay_batched(f(S[l]), f(q[l]), f(k[l]), f(v[l]), f(g[l]), f(beta[l]),
                                                     n_acc.cpu().numpy())
        assert rel(S_new[l], S_ref) < TOL_F32 and rel(out[l], out_ref) < tol_out
