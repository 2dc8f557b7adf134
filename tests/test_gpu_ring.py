"""GPU raw-input ring against the oracle ring: pushes, FIFO overwrite, window layout, and the
replay of the accepted prefix straight from the ring."""
import numpy as np
import pytest
import torch

from kda_delta_rule_gb300 import inputs as I
from oracle import kda_oracle as O
from parity import TOL_BF16_STORED_OUT, TOL_F32, rel

pytestmark = pytest.mark.gpu
f = I.to_f64_numpy


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


@pytest.mark.parametrize("dtype,dk,dv,mode", [(torch.float32, 32, 32, 0), (torch.bfloat16, 128, 64, 1)])
@pytest.mark.parametrize("pushes", [3, 6])
def test_ring_matches_oracle_and_plain_replay(K, dtype, dk, dv, mode, pushes):
    B, H, cap = 5, 3, 4
    S, proj, n_acc = I.replay_inputs(B, H, dk, dv, pushes, dtype=dtype, seed=11 + pushes, state_std=0.1)
    pr = proj.to("cuda")
    ring = K.RawInputRing(cap, B, H, dk, dv, dtype=dtype)
    ref = O.RawInputRing(cap)
    sizes = []
    for t in range(pushes):
        ring.push(pr.q[t], pr.k[t], pr.v[t], pr.g[t], pr.beta[t])
        ref.push(f(proj.q[t]), f(proj.k[t]), f(proj.v[t]), f(proj.g[t]), f(proj.beta[t]))
        sizes.append(len(ring))
    assert sizes == [min(t + 1, cap) for t in range(pushes)]
    win = ring.window()
    torch.cuda.synchronize()
    for got, want in zip(win, ref.window()):          # the stored values, oldest first
        assert np.array_equal(f(got), want)
    Sc = S.cuda()
    snap = Sc.clone()
    n = torch.clamp(n_acc, max=len(ring)).to(torch.int32).cuda()
    S_new, out = ring.verify_replay(Sc, n, mode=mode)
    S_plain, out_plain = K.kda_verify_replay(Sc, *[w.contiguous() for w in win], n, mode=mode)
    torch.cuda.synchronize()
    assert torch.equal(Sc, snap), "the committed state was written"
    assert torch.equal(S_new, S_plain) and torch.equal(out, out_plain)
    S_ref, out_ref = O.verify_and_replay_batched(f(S), *ref.window(), n.cpu().numpy(), mode)
    assert rel(S_new, S_ref) < TOL_F32
    assert rel(out, out_ref) < (TOL_F32 if dtype == torch.float32 else TOL_BF16_STORED_OUT)
    ring.reset()
    assert len(ring) == 0
