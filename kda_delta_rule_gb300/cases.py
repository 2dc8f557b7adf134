"""Run one KDA workload a few times on cuda:0 (for profilers and quick timing).

    python -m kda_delta_rule_gb300.cases decode   [--reps N]   # B=256 H=32 d=128, bf16 projections
    python -m kda_delta_rule_gb300.cases replay   [--reps N]   # B=32 H=16 d=32 draft 8, fp32
    python -m kda_delta_rule_gb300.cases replay_layers [--reps N]   # the same for 64 stacked layers, one launch
    python -m kda_delta_rule_gb300.cases prefill  [--reps N]   # T=8192 H=32 d=128 bf16, 16 checkpoints
    python -m kda_delta_rule_gb300.cases varlen   [--reps N]   # 64 seqs, ~0.5M tokens, H=32 d=128 bf16
    python -m kda_delta_rule_gb300.cases pack     [--reps N]   # pack+unpack of a (256,32,128,128) state
    python -m kda_delta_rule_gb300.cases layer    [--reps N]   # kda_input_prep then prefill, T=8192 H=32 d=128
    python -m kda_delta_rule_gb300.cases prologue [--reps N]   # kda_input_prep alone, T=8192 H=32 d=128 bf16
    python -m kda_delta_rule_gb300.cases decode_vk    [--reps N]   # decode on 256 of 512 transposed pool slots
    python -m kda_delta_rule_gb300.cases decode_fused [--reps N]   # decode with the input prologue, B=256
    python -m kda_delta_rule_gb300.cases scan     [--reps N]   # sequence-parallel prefill, T=65536 H=4 d=128
    python -m kda_delta_rule_gb300.cases scan32   [--reps N]   # the same at T=8192 H=32 d=128, 4 pieces

Each case prints the mean device time per call measured with CUDA events.
"""
from __future__ import annotations

import argparse

import torch

from . import inputs as I
from . import kda as K


def _time(fn, reps):
    fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def case_decode(reps, H=32, d=128, B=256):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    S = (0.05 * torch.randn(B, H, d, d, generator=gen, device="cuda")).contiguous()
    p = I.decode_step_projections(B, H, d, d, dtype=torch.bfloat16, seed=1, device="cuda")
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    return _time(lambda: K.kda_decode_step(S, p["q"], p["k"], p["v"], p["g"], p["beta"], o=o), reps)


def case_replay(reps):
    S, pr, n = I.replay_inputs(32, 16, 32, 32, 8, dtype=torch.float32, seed=0, device="cuda")
    S_new = torch.empty_like(S)
    out = torch.empty(32, 16, 8, 32, device="cuda")
    return _time(lambda: K.kda_verify_replay(S, pr.q, pr.k, pr.v, pr.g, pr.beta, n, S_new=S_new, out=out),
                 reps)


def case_replay_layers(reps, layers=64):
    """64 stacked KDA layers of the replay shape, each with its own state and draft
    projections and the accepted counts shared, in one kda_verify_replay_layers launch."""
    sets = [I.replay_inputs(32, 16, 32, 32, 8, dtype=torch.float32, seed=i, device="cuda") for i in range(layers)]
    n = sets[0][2].to("cuda")
    S = torch.stack([x[0] for x in sets])
    pj = {nm: torch.stack([getattr(x[1], nm) for x in sets]) for nm in ("q", "k", "v", "g", "beta")}
    del sets
    S_new = torch.empty_like(S)
    out = torch.empty(layers, 32, 16, 8, 32, device="cuda")
    return _time(lambda: K.kda_verify_replay_layers(S, pj["q"], pj["k"], pj["v"], pj["g"], pj["beta"], n,
                                                    S_new=S_new, out=out), reps)


def _prefill(lengths, reps, H=32, d=128, stride=512):
    S0, p, cu = I.prefill_inputs(lengths, H, d, d, dtype=torch.bfloat16, seed=0, device="cuda")
    n_ck = K.kda_num_checkpoints(cu, cu[-1], stride)
    pool = K.PagePool(H * d * d * 4, n_ck)
    ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device="cuda")
    o = torch.empty(cu[-1], H, d, dtype=torch.bfloat16, device="cuda")
    Sf = torch.empty_like(S0)
    ws = torch.empty(max(K.kda_prefill_workspace_bytes(cu, cu[-1], H, d, d, torch.bfloat16), 16),
                     dtype=torch.uint8, device="cuda")
    return _time(lambda: K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                                               ckpt_stride=stride, page_pool=pool, ckpt_page_ids=ids,
                                               o=o, S_final=Sf, workspace=ws), reps)


def case_prefill(reps):
    return _prefill([8192], reps)


def case_varlen(reps):
    return _prefill(I.varlen_lengths(64, seed=0), reps)


def case_pack(reps):
    S = torch.randn(256, 32, 128, 128, device="cuda")
    flat = torch.empty(S.numel(), device="cuda")
    back = torch.empty_like(S)

    def run():
        K.kda_pack_heads(S, flat=flat)
        K.kda_unpack_heads(flat, back)
    return _time(run, reps)


def case_layer(reps, T=8192, H=32, d=128, w=4):
    raw, cu = I.prologue_inputs([T], H, d, d, w=w, dtype=torch.bfloat16, seed=0, device="cuda")
    S0, _, _ = I.prefill_inputs([T], H, d, d, dtype=torch.bfloat16, seed=1, device="cuda")
    p = K.kda_input_prep(raw["mixed"], raw["weight"], raw["g_logits"], raw["beta_logits"], window_in=raw["window"])
    pool = K.PagePool(H * d * d * 4, T // 512)
    ids = torch.tensor(pool.alloc(T // 512), dtype=torch.int32, device="cuda")
    o = torch.empty(T, H, d, dtype=torch.bfloat16, device="cuda")
    Sf = torch.empty_like(S0)
    ws = torch.empty(K.kda_prefill_workspace_bytes(cu, T, H, d, d, torch.bfloat16), dtype=torch.uint8, device="cuda")

    def run():
        K.kda_input_prep(raw["mixed"], raw["weight"], raw["g_logits"], raw["beta_logits"], window_in=raw["window"],
                         out=p)
        K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu, ckpt_stride=512,
                              page_pool=pool, ckpt_page_ids=ids, o=o, S_final=Sf, workspace=ws)
    return _time(run, reps)


def case_prologue(reps, T=8192, H=32, d=128, w=4):
    raw, _ = I.prologue_inputs([T], H, d, d, w=w, dtype=torch.bfloat16, seed=0, device="cuda")
    p = K.kda_input_prep(raw["mixed"], raw["weight"], raw["g_logits"], raw["beta_logits"], window_in=raw["window"])
    return _time(lambda: K.kda_input_prep(raw["mixed"], raw["weight"], raw["g_logits"], raw["beta_logits"],
                                          window_in=raw["window"], out=p), reps)


def case_decode_vk(reps, H=32, d=128, B=256):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    pool = (0.05 * torch.randn(2 * B, H, d, d, generator=gen, device="cuda")).contiguous()
    slots = torch.randperm(2 * B, generator=gen, device="cuda")[:B].to(torch.int32)
    p = I.decode_step_projections(B, H, d, d, dtype=torch.bfloat16, seed=1, device="cuda")
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    return _time(lambda: K.kda_decode_step_slots(pool, slots, p["q"], p["k"], p["v"], p["g"], p["beta"], o=o,
                                                 layout=K.LAYOUT_VK), reps)


def case_decode_fused(reps, H=32, d=128, B=256, w=4):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    S = (0.05 * torch.randn(B, H, d, d, generator=gen, device="cuda")).contiguous()
    raw, _ = I.prologue_inputs([1] * B, H, d, d, w=w, dtype=torch.bfloat16, seed=2, device="cuda")
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    return _time(lambda: K.kda_decode_step_fused(S, raw["window"], raw["mixed"], raw["weight"], raw["g_logits"],
                                                 raw["beta_logits"], o=o), reps)


def case_scan(reps, T=65536, H=4, d=128, segments=0):
    S0, p, cu = I.prefill_inputs([T], H, d, d, dtype=torch.bfloat16, seed=0, device="cuda")
    ws = torch.empty(K.kda_prefill_scan_workspace_bytes(T, H, d, d, torch.bfloat16, 0, segments), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty(T, H, d, dtype=torch.bfloat16, device="cuda")
    Sf = torch.empty_like(S0)
    return _time(lambda: K.kda_prefill_scan(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], ckpt_stride=0, o=o,
                                            S_final=Sf, segments=segments, workspace=ws), reps)


def case_scan32(reps):
    """The sequence-parallel path at the long-prefill shape (T=8192, H=32), four pieces."""
    return case_scan(reps, T=8192, H=32, segments=4)


CASES = {"scan": case_scan, "scan32": case_scan32, "decode": case_decode, "replay": case_replay,
         "replay_layers": case_replay_layers, "prefill": case_prefill,
         "varlen": case_varlen, "pack": case_pack, "layer": case_layer, "prologue": case_prologue, "decode_vk": case_decode_vk,
         "decode_fused": case_decode_fused}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    ms = CASES[args.case](args.reps)
    print(f"{args.case}: {ms:.4f} ms per call (mean of {args.reps})")


if __name__ == "__main__":
    main()
