"""The hot-path calls captured in a CUDA graph and replayed give the same bits as the eager calls
(the chain kernel is a programmatic dependent of the prep; the step kernels launch that way on
eager streams only)."""
import pytest
import torch

from kda_delta_rule_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    from kda_delta_rule_gb300 import kda
    return kda


def test_prefill_in_a_graph_is_bit_identical(K):
    """Two sequences (512 and 200 tokens), H=2, dk=dv=128, bf16, checkpoints every 128 tokens."""
    H, d, stride = 2, 128, 128
    S0, p, cu = I.prefill_inputs([512, 200], H, d, d, dtype=torch.bfloat16, seed=41, device="cuda")
    T = cu[-1]
    n_ck = K.kda_num_checkpoints(cu, T, stride)
    ws = torch.empty(K.kda_prefill_workspace_bytes(cu, T, H, d, d, torch.bfloat16), dtype=torch.uint8, device="cuda")
    runs = []
    for graph in (False, True):
        pool = K.PagePool(H * d * d * 4, n_ck)
        ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device="cuda")
        pos = torch.full((n_ck,), -1, dtype=torch.int32, device="cuda")
        o = torch.empty(T, H, d, dtype=torch.bfloat16, device="cuda")
        Sf = torch.empty_like(S0)

        def call():
            K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu, ckpt_stride=stride,
                                  o=o, S_final=Sf, page_pool=pool, ckpt_page_ids=ids, ckpt_pos=pos, workspace=ws)

        call()                                   # eager (and the warm-up before a capture)
        torch.cuda.synchronize()
        if graph:
            o.zero_(), Sf.zero_(), pool.arena.zero_(), pos.fill_(-1)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            g.replay()
            g.replay()
        torch.cuda.synchronize()
        runs.append((o.clone(), Sf.clone(), torch.stack([pool.page(int(i)) for i in ids]), pos.clone()))
    assert K.kda_device_errors() == 0
    for a, b in zip(*runs):
        assert torch.equal(a, b)


def test_replay_and_decode_in_a_graph_are_bit_identical(K):
    """Replay B=8, H=4, dk=dv=32, draft 8 (fp32), then decode B=4, H=2, dk=dv=128 (bf16
    projections): graph replays equal the eager calls."""
    B, H, d, draft = 8, 4, 32, 8
    Sc, pr, na = I.replay_inputs(B, H, d, d, draft, dtype=torch.float32, seed=5, device="cuda")
    outs = []
    for graph in (False, True):
        Sn = torch.empty_like(Sc)
        out = torch.empty(B, H, draft, d, dtype=torch.float32, device="cuda")

        def call():
            K.kda_verify_replay(Sc, pr.q, pr.k, pr.v, pr.g, pr.beta, na, S_new=Sn, out=out)

        call()
        torch.cuda.synchronize()
        if graph:
            Sn.zero_(), out.zero_()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            g.replay()
        torch.cuda.synchronize()
        outs.append((Sn.clone(), out.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])

    B, H, d = 4, 2, 128
    S0, p = I.decode_inputs(B, H, d, d, dtype=torch.bfloat16, seed=9, device="cuda")
    res = []
    for graph in (False, True):
        S = S0.clone()
        o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")

        def step(state):
            K.kda_decode_step(state, p["q"], p["k"], p["v"], p["g"], p["beta"], o=o)

        if graph:
            step(S0.clone())                     # warm-up on a copy: S itself takes both steps in the graph
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(S)
            g.replay()
            g.replay()
        else:
            step(S)
            step(S)
        torch.cuda.synchronize()
        res.append((S.clone(), o.clone()))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
