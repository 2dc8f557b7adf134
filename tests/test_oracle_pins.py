"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

None of these compares the oracle with a retyped copy of itself: each check is
a hand-derived value, a closed form, an independent formulation (explicit
transition-matrix products), a value the pages print, or an invariant.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import kda_oracle as O
from kda_delta_rule_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_printed_values.json")
f64 = I.to_f64_numpy


def _rand_head(T, dk, dv, seed, g_min=-5.0, S_std=0.3):
    S0, p, _ = I.prefill_inputs(T, 1, dk, dv, dtype=torch.float64, seed=seed,
                                state_std=S_std, g_min=g_min)
    a = {n: f64(t)[:, 0] for n, t in p.items()}
    return f64(S0)[0, 0], a


# --------------------------------------------------------------------------
# Hand-derived scalar examples (dk = dv = 1)
# --------------------------------------------------------------------------

def test_scalar_step_by_hand():
    # S0 = 1, k = q = 1, v = 2, e^g = 1/2, beta = 1/2.
    # decay first: S' = 0.5, delta = 2 - 0.5 = 1.5, S = 0.5 + 0.5*1.5 = 1.25, o = 1.25
    # undecayed delta: delta = 2 - 1 = 1, S = 0.5 + 0.5*1 = 1.0, o = 1.0
    args = (np.array([[1.0]]), np.array([1.0]), np.array([1.0]), np.array([2.0]),
            np.array([math.log(0.5)]), np.array(0.5))
    o, S = O.kda_step(*args, mode=O.DECAY_FIRST)
    assert S[0, 0] == pytest.approx(1.25, abs=1e-15) and o[0] == pytest.approx(1.25, abs=1e-15)
    o, S = O.kda_step(*args, mode=O.UNDECAYED_DELTA)
    assert S[0, 0] == pytest.approx(1.0, abs=1e-15) and o[0] == pytest.approx(1.0, abs=1e-15)


def test_two_by_two_step_by_hand():
    # dk = dv = 2, S0 = I, k = (0.6, 0.8), q = (1, 0), v = (1, -1), g = (0, ln 0.5), beta = 1.
    # decay first: S' = diag(1, .5); S'^T k = (0.6, 0.4); delta = (0.4, -1.4)
    #   S = S' + k delta^T = [[1.24, -0.84], [0.32, -0.62]]; o = row 0 = (1.24, -0.84)
    # undecayed: S^T k = (0.6, 0.8); delta = (0.4, -1.8)
    #   S = diag(1,.5) + k delta^T = [[1.24, -1.08], [0.32, -0.94]]; o = (1.24, -1.08)
    S0 = np.eye(2)
    k = np.array([0.6, 0.8]); q = np.array([1.0, 0.0]); v = np.array([1.0, -1.0])
    g = np.array([0.0, math.log(0.5)]); beta = np.array(1.0)
    o, S = O.kda_step(S0, q, k, v, g, beta, O.DECAY_FIRST)
    np.testing.assert_allclose(S, [[1.24, -0.84], [0.32, -0.62]], atol=1e-14)
    np.testing.assert_allclose(o, [1.24, -0.84], atol=1e-14)
    o, S = O.kda_step(S0, q, k, v, g, beta, O.UNDECAYED_DELTA)
    np.testing.assert_allclose(S, [[1.24, -1.08], [0.32, -0.94]], atol=1e-14)
    np.testing.assert_allclose(o, [1.24, -1.08], atol=1e-14)
    assert np.array_equal(S0, np.eye(2))           # the input state is not modified


# --------------------------------------------------------------------------
# Brute force: explicit products of the dk x dk transitions, tiny T
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", [O.DECAY_FIRST, O.UNDECAYED_DELTA])
@pytest.mark.parametrize("T,dk,dv,seed", [(1, 3, 2, 0), (2, 4, 3, 1), (3, 5, 4, 2), (3, 2, 6, 3)])
def test_recurrent_equals_unrolled_products(mode, T, dk, dv, seed):
    S0, a = _rand_head(T, dk, dv, seed)
    o_ref, S_ref = O.unrolled_products(S0, a["q"], a["k"], a["v"], a["g"], a["beta"], mode)
    o, S = O.kda_recurrent(S0, a["q"], a["k"], a["v"], a["g"], a["beta"], mode)
    np.testing.assert_allclose(o, o_ref, atol=1e-13, rtol=0)
    np.testing.assert_allclose(S, S_ref, atol=1e-13, rtol=0)


# --------------------------------------------------------------------------
# Closed forms and special cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", [O.DECAY_FIRST, O.UNDECAYED_DELTA])
def test_beta_zero_is_pure_decay(mode):
    T, dk, dv = 7, 6, 5
    S0, a = _rand_head(T, dk, dv, 11)
    beta = np.zeros(T)
    o, S, states = O.kda_recurrent(S0, a["q"], a["k"], a["v"], a["g"], beta, mode,
                                   return_states=True)
    cum = np.cumsum(a["g"], axis=0)
    for t in range(T):
        S_t = np.exp(cum[t])[:, None] * S0
        np.testing.assert_allclose(states[t + 1], S_t, atol=1e-14)
        np.testing.assert_allclose(o[t], S_t.T @ a["q"][t], atol=1e-14)


def test_zero_gate_modes_coincide_and_equal_plain_delta_rule():
    # g = 0: both orderings reduce to S_t = (I - beta k k^T) S_{t-1} + beta k v^T.
    T, dk, dv = 9, 5, 4
    S0, a = _rand_head(T, dk, dv, 12)
    g0 = np.zeros_like(a["g"])
    o0, S0_ = O.kda_recurrent(S0, a["q"], a["k"], a["v"], g0, a["beta"], O.DECAY_FIRST)
    o1, S1_ = O.kda_recurrent(S0, a["q"], a["k"], a["v"], g0, a["beta"], O.UNDECAYED_DELTA)
    np.testing.assert_allclose(o0, o1, atol=1e-14)
    np.testing.assert_allclose(S0_, S1_, atol=1e-14)
    S = S0.copy()
    for t in range(T):
        k = a["k"][t]
        S = (np.eye(dk) - a["beta"][t] * np.outer(k, k)) @ S + a["beta"][t] * np.outer(k, a["v"][t])
        np.testing.assert_allclose(o0[t], S.T @ a["q"][t], atol=1e-13)
    np.testing.assert_allclose(S0_, S, atol=1e-13)


def test_decay_first_perfect_write_and_page1_breaks_it():
    # beta = 1, |k| = 1: decay first gives S_t^T k_t = v_t exactly (the write
    # fully corrects the decayed prediction).  The undecayed-delta ordering
    # does not when g != 0, which tells the two orderings apart.
    T, dk, dv = 6, 8, 5
    S0, a = _rand_head(T, dk, dv, 13)
    ones = np.ones(T)
    _, _, st = O.kda_recurrent(S0, a["q"], a["k"], a["v"], a["g"], ones, O.DECAY_FIRST,
                               return_states=True)
    for t in range(T):
        np.testing.assert_allclose(st[t + 1].T @ a["k"][t], a["v"][t], atol=1e-13)
    _, _, st1 = O.kda_recurrent(S0, a["q"], a["k"], a["v"], a["g"], ones, O.UNDECAYED_DELTA,
                                return_states=True)
    worst = max(np.abs(st1[t + 1].T @ a["k"][t] - a["v"][t]).max() for t in range(T))
    assert worst > 1e-3


def test_cold_start_single_token():
    # S0 = 0, T = 1: o = beta (k . q) v in both orderings.
    dk, dv = 7, 3
    _, a = _rand_head(1, dk, dv, 14)
    for mode in (O.DECAY_FIRST, O.UNDECAYED_DELTA):
        o, S = O.kda_step(np.zeros((dk, dv)), a["q"][0], a["k"][0], a["v"][0], a["g"][0],
                          a["beta"][0], mode)
        np.testing.assert_allclose(o, a["beta"][0] * (a["k"][0] @ a["q"][0]) * a["v"][0],
                                   atol=1e-15)
        np.testing.assert_allclose(S, a["beta"][0] * np.outer(a["k"][0], a["v"][0]), atol=1e-15)


def test_ut_inverse_is_the_inverse():
    rng = np.random.default_rng(3)
    A = np.tril(rng.standard_normal((12, 12)) * 0.3, -1)
    T = O.ut_inverse(A)
    np.testing.assert_allclose(T @ (np.eye(12) + A), np.eye(12), atol=1e-12)
    np.testing.assert_allclose(T, np.linalg.inv(np.eye(12) + A), atol=1e-12)


# --------------------------------------------------------------------------
# Chunked WY/UT form == token recurrence (an independent algorithm)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", [O.DECAY_FIRST, O.UNDECAYED_DELTA])
@pytest.mark.parametrize("T,chunk", [(64, 64), (200, 64), (131, 16), (5, 64), (96, 32)])
def test_chunked_equals_recurrent(mode, T, chunk):
    S0, p, cu = I.prefill_inputs(T, 2, 12, 6, dtype=torch.float64, seed=T + chunk)
    args = [f64(S0)] + [f64(p[n]) for n in ("q", "k", "v", "g", "beta")]
    oc, Sc, cc = O.prefill_chunked(*args, cu_seqlens=cu, chunk=chunk, ckpt_stride=chunk, mode=mode)
    orr, Sr, cr = O.prefill_recurrent(*args, cu_seqlens=cu, ckpt_stride=chunk, mode=mode)
    scale = max(1.0, np.abs(orr).max())
    assert np.abs(oc - orr).max() <= 1e-10 * scale
    assert np.abs(Sc - Sr).max() <= 1e-10
    assert [(n, t) for n, t, _ in cc] == [(n, t) for n, t, _ in cr]
    for (_, _, a), (_, _, b) in zip(cc, cr):
        assert np.abs(a - b).max() <= 1e-10


def test_chunked_strong_decay_no_overflow():
    # Cumulative log-decay over a 64-token chunk reaches about -300 here; any
    # factorisation e^{Gamma_r} * e^{-Gamma_s} would overflow fp32 (and near fp64).
    T = 128
    S0, p, cu = I.prefill_inputs(T, 1, 8, 4, dtype=torch.float64, seed=5, g_min=-9.0)
    args = [f64(S0)] + [f64(p[n]) for n in ("q", "k", "v", "g", "beta")]
    assert np.cumsum(args[4][:64, 0], axis=0).min() < -200
    oc, Sc, _ = O.prefill_chunked(*args, cu_seqlens=cu, chunk=64, ckpt_stride=64)
    orr, Sr, _ = O.prefill_recurrent(*args, cu_seqlens=cu, ckpt_stride=64)
    assert np.isfinite(oc).all() and np.isfinite(Sc).all()
    assert np.abs(oc - orr).max() <= 1e-10 and np.abs(Sc - Sr).max() <= 1e-10


def test_varlen_is_independent_sequences():
    lengths = [64, 128, 37, 0, 192]
    S0, p, cu = I.prefill_inputs(lengths, 2, 8, 4, dtype=torch.float64, seed=21)
    args = [f64(S0)] + [f64(p[n]) for n in ("q", "k", "v", "g", "beta")]
    o, S, ck = O.prefill_chunked(*args, cu_seqlens=cu, chunk=64, ckpt_stride=64)
    for n, L in enumerate(lengths):
        a, b = cu[n], cu[n + 1]
        sl = [args[0][n:n + 1]] + [x[a:b] for x in args[1:]]
        o1, S1, ck1 = O.prefill_recurrent(*sl, cu_seqlens=None, ckpt_stride=64)
        np.testing.assert_allclose(o[a:b], o1, atol=1e-10)
        np.testing.assert_allclose(S[n], S1[0], atol=1e-10)
        mine = [(t, s) for m, t, s in ck if m == n]
        assert [t for t, _ in mine] == [t for _, t, _ in ck1]
    np.testing.assert_array_equal(S[3], args[0][3])    # an empty sequence keeps S0


# --------------------------------------------------------------------------
# Checkpoint boundaries
# --------------------------------------------------------------------------

def test_checkpoint_positions_long_prefill():
    # T = 8192, stride 512: 16 boundaries 512..8192, the last one at T itself.
    pos = O.checkpoint_positions(8192, 512)
    assert pos == [512 * j for j in range(1, 17)]
    assert O.checkpoint_positions(511, 512) == []
    assert O.checkpoint_positions(1000, 512) == [512]
    assert O.num_checkpoints([8192, 1000, 511, 1024], 512) == 16 + 1 + 0 + 2


def test_last_checkpoint_is_final_state_bitwise():
    S0, p, cu = I.prefill_inputs(256, 2, 8, 4, dtype=torch.float64, seed=9)
    args = [f64(S0)] + [f64(p[n]) for n in ("q", "k", "v", "g", "beta")]
    o, S, ck = O.prefill_chunked(*args, cu_seqlens=cu, chunk=64, ckpt_stride=128)
    assert [t for _, t, _ in ck] == [128, 256]
    assert np.array_equal(ck[-1][2], S[0])


# --------------------------------------------------------------------------
# Replay: the pages' three acceptance scenarios and the clone invariant
# --------------------------------------------------------------------------

def _golden():
    with open(GOLDEN) as fh:
        return json.load(fh)


@pytest.mark.parametrize("mode", [O.DECAY_FIRST, O.UNDECAYED_DELTA])
def test_replay_scenarios_match_recurrent(mode):
    gold = _golden()
    draft = gold["acceptance_scenarios"]["draft"]
    B, H, dk, dv = 2, 3, 8, 8
    S, proj, _ = I.replay_inputs(B, H, dk, dv, draft, dtype=torch.float64, seed=4)
    S = f64(S)
    P = {n: f64(getattr(proj, n)) for n in ("q", "k", "v", "g", "beta")}
    o_full, _, states = O.kda_recurrent(S, P["q"], P["k"], P["v"], P["g"], P["beta"], mode,
                                        return_states=True)
    for n in gold["acceptance_scenarios"]["n_accepted"]:
        S_before = S.copy()
        S_new, out = O.verify_and_replay(S, P["q"], P["k"], P["v"], P["g"], P["beta"], n, mode)
        assert out.shape == (B, H, n, dv)
        assert np.array_equal(S, S_before)                      # committed state untouched
        bound = gold["replay_vs_recurrent"]["bound_fp64"]
        if n:
            assert np.abs(out - np.moveaxis(o_full[:n], 0, 2)).max() < bound
        assert np.abs(S_new - states[n]).max() < bound
        if n == 0:
            assert np.array_equal(S_new, S)


def test_batched_replay_zero_pads_and_matches_per_sequence():
    B, H, dk, dv, draft = 5, 2, 4, 3, 6
    S, proj, n_acc = I.replay_inputs(B, H, dk, dv, draft, dtype=torch.float64, seed=8,
                                     n_accepted=[0, 6, 3, 1, 6])
    P = {n: f64(getattr(proj, n)) for n in ("q", "k", "v", "g", "beta")}
    S_new, out = O.verify_and_replay_batched(f64(S), P["q"], P["k"], P["v"], P["g"], P["beta"],
                                             n_acc.numpy())
    for b, n in enumerate([0, 6, 3, 1, 6]):
        o, Sb = O.kda_recurrent(f64(S)[b], P["q"][:n, b], P["k"][:n, b], P["v"][:n, b],
                                P["g"][:n, b], P["beta"][:n, b])
        np.testing.assert_allclose(out[b, :, :n], np.moveaxis(o, 0, 1), atol=1e-15)
        assert np.all(out[b, :, n:] == 0.0)
        np.testing.assert_allclose(S_new[b], Sb, atol=1e-15)


def test_replay_counts_clamp_to_the_draft():
    """An accepted count counts draft tokens, so it lies in [0, draft] ([SERVE] §1.2); counts
    outside are clamped: a negative count replays nothing (state unchanged, zero rows), a count
    past the draft replays all of it (the recurrence over the whole draft)."""
    B, H, dk, dv, draft = 3, 2, 4, 3, 5
    S, proj, _ = I.replay_inputs(B, H, dk, dv, draft, dtype=torch.float64, seed=9)
    S = f64(S)
    P = {n: f64(getattr(proj, n)) for n in ("q", "k", "v", "g", "beta")}
    S_new, out = O.verify_and_replay_batched(S, P["q"], P["k"], P["v"], P["g"], P["beta"],
                                             np.array([-2, draft + 3, draft]))
    assert np.array_equal(S_new[0], S[0]) and np.all(out[0] == 0.0)
    for b in (1, 2):
        o, Sb = O.kda_recurrent(S[b], P["q"][:, b], P["k"][:, b], P["v"][:, b], P["g"][:, b], P["beta"][:, b])
        np.testing.assert_allclose(out[b], np.moveaxis(o, 0, 1), atol=1e-15)
        np.testing.assert_allclose(S_new[b], Sb, atol=1e-15)


def test_draft_window_layout():
    # Tab 4 panel b: (draft=3, B=1, H=2, D=3), step i filled with i.
    lay = _golden()["draft_window_layout"]
    q = torch.stack([torch.full((lay["B"], lay["H"], lay["D"]), float(i)) for i in range(lay["draft"])])
    proj = I.DraftProjections(q, q, q, q, q[..., 0])
    assert tuple(proj.q.shape) == (3, 1, 2, 3) and proj.draft == 3
    for i in range(3):
        assert torch.all(proj.q[i] == i)


def _ring_step(rng, B, H, dk, dv):
    q, k = rng.normal(size=(B, H, dk)), rng.normal(size=(B, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return (q, k, rng.normal(size=(B, H, dv)), -5.0 / (1.0 + np.exp(-rng.normal(size=(B, H, dk)))),
            1.0 / (1.0 + np.exp(-rng.normal(size=(B, H)))))


def test_ring_window_sizes_printed():
    # Tab 4 panel a: capacity 4, sizes 1, 2, 3, then 4 from push(3) on.
    gold = _golden()["ring_window_sizes"]
    ring = O.RawInputRing(gold["capacity"])
    sizes = []
    rng = np.random.default_rng(0)
    for _ in gold["sizes_after_push"]:
        ring.push(*_ring_step(rng, 1, 1, 2, 2))
        sizes.append(len(ring))
    assert sizes == gold["sizes_after_push"]


def test_ring_window_layout_printed():
    # Tab 4 panel b: window() of three pushes is (draft=3, B=1, H=2, D=3), row i holds i.
    lay = _golden()["draft_window_layout"]
    ring = O.RawInputRing(4)
    for i in range(lay["draft"]):
        x = np.full((lay["B"], lay["H"], lay["D"]), float(i))
        ring.push(x, x, x, x, x[..., 0])
    q, k, v, g, beta = ring.window()
    assert q.shape == (3, 1, 2, 3) and beta.shape == (3, 1, 2)
    for i in range(3):
        assert np.all(q[i] == i) and np.all(beta[i] == i)


def test_ring_overwrites_oldest_first():
    rng = np.random.default_rng(1)
    steps = [_ring_step(rng, 2, 3, 4, 5) for _ in range(6)]
    ring = O.RawInputRing(4)
    for st in steps:
        ring.push(*st)
    win = ring.window()
    for j in range(4):                     # pushes 2, 3, 4, 5 in push order
        for t in range(5):
            assert np.array_equal(win[t][j], steps[2 + j][t])
    ring.reset()
    assert len(ring) == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_ring_replay_equals_recurrent(mode):
    # Tab 4 panel c: replay from the window == the recurrence over the same steps, error 0.
    gold = _golden()["ring_replay_error"]
    rng = np.random.default_rng(2)
    B, H, dk, dv = 2, 2, 4, 3
    S0 = rng.normal(size=(B, H, dk, dv))
    steps = [_ring_step(rng, B, H, dk, dv) for _ in range(6)]
    ring = O.RawInputRing(4)
    for st in steps:
        ring.push(*st)
    q, k, v, g, beta = ring.window()
    S_new, out = O.verify_and_replay(S0, q, k, v, g, beta, 3, mode)
    S = S0.copy()
    outs = []
    for j in range(3):                     # the oldest held step is push 2
        o, S = O.kda_step(S, *steps[2 + j], mode)
        outs.append(o)
    assert np.max(np.abs(S_new - S)) == gold["max_abs_error"]
    assert np.max(np.abs(out - np.stack(outs, axis=-2))) == gold["max_abs_error"]


# --------------------------------------------------------------------------
# Page packing
# --------------------------------------------------------------------------

def test_pack_layout_and_roundtrip():
    B, H, dk, dv = 2, 3, 4, 5
    S = np.random.default_rng(0).standard_normal((B, H, dk, dv))
    flat = O.pack_heads(S)
    for b, h, i, j in [(0, 0, 0, 0), (1, 2, 3, 4), (0, 2, 1, 3), (1, 0, 3, 0)]:
        assert flat[((b * H + h) * dk + i) * dv + j] == S[b, h, i, j]
    back = O.unpack_heads(flat, B, H, dk, dv)
    assert np.array_equal(back, S)
    assert np.abs(back - S).max() < _golden()["pack_roundtrip"]["bound_fp64"]


def test_store_load_zero_padded_page():
    S = np.random.default_rng(1).standard_normal((1, 2, 3, 4))
    page = O.store_kda(S, 40)
    assert page.size == 40 and np.all(page[24:] == 0.0)
    assert np.array_equal(O.load_kda(page, 1, 2, 3, 4), S)
    with pytest.raises(ValueError):
        O.store_kda(S, 23)


# --------------------------------------------------------------------------
# Byte accounting
# --------------------------------------------------------------------------

def test_snapshot_cost_ratio_printed_values():
    for row in _golden()["snapshot_cost_ratio"]:
        r = O.snapshot_cost_ratio(row["H"], row["dk"], row["dv"])
        if row["consistent"]:
            assert round(r, row["digits"]) == row["printed"], row
        else:
            # page error: the closed form gives 1024/129, not the printed 4.0
            assert r == pytest.approx(1024 / 129) and round(r, 1) != row["printed"]


def test_snapshot_cost_ratio_properties():
    # > 1 and growing with the state size; independent of draft length and dtype.
    rs = [O.snapshot_cost_ratio(4, d, d) for d in (8, 16, 32, 64, 128)]
    assert all(r > 1 for r in rs) and all(a < b for a, b in zip(rs, rs[1:]))
    for draft in (1, 2, 8, 32):
        for item in (2, 4, 8):
            snap = draft * O.snapshot_bytes_per_step(16, 32, 32, item)
            proj = draft * O.projection_bytes_per_step(16, 32, 32, item)
            assert snap / proj == pytest.approx(O.snapshot_cost_ratio(16, 32, 32))


# --------------------------------------------------------------------------
# Input prologue: ShortConv, activation, L2Norm, gates from logits
# --------------------------------------------------------------------------
def _prologue(T, H=2, dk=4, dv=3, w=4, seed=0):
    p, _ = I.prologue_inputs([T], H, dk, dv, w=w, dtype=torch.float64, seed=seed)
    return {n: f64(t) for n, t in p.items()}


@pytest.mark.parametrize("w", [2, 3, 4])
def test_short_conv_is_numpy_correlation(w):
    """A causal depthwise conv over [window; x] is, channel by channel, numpy's valid
    cross-correlation with the channel's taps (an independent library routine)."""
    p = _prologue(11, w=w, seed=w)
    x, W, win = p["mixed"], p["weight"], p["window"][0]
    y, win_out = O.short_conv(x, W, win)
    z = np.concatenate([win, x])
    for c in range(x.shape[1]):
        assert np.allclose(y[:, c], np.correlate(z[:, c], W[c], mode="valid"), rtol=0, atol=1e-12)
    assert np.array_equal(win_out, z[-(w - 1):])


def test_short_conv_newest_and_oldest_taps():
    """Only the newest tap set: the input itself. Only the oldest: the input w - 1
    rows earlier, i.e. the window first."""
    p = _prologue(7, w=4, seed=3)
    x, win = p["mixed"], p["window"][0]
    C = x.shape[1]
    newest = np.zeros((C, 4)); newest[:, 3] = 1.0
    oldest = np.zeros((C, 4)); oldest[:, 0] = 1.0
    assert np.array_equal(O.short_conv(x, newest, win)[0], x)
    y = O.short_conv(x, oldest, win)[0]
    assert np.array_equal(y[:3], win) and np.array_equal(y[3:], x[:4])
    assert np.array_equal(O.short_conv(x, oldest)[0][:3], np.zeros((3, C)))   # fresh sequence


def test_activation_and_sigmoid_closed_forms():
    assert O.sigmoid(0.0) == 0.5
    assert O.silu(0.0) == 0.0
    assert O.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), abs=1e-15)
    assert O.silu(-2.0) == pytest.approx(-2.0 / (1.0 + math.exp(2.0)), abs=1e-15)
    assert O.silu(40.0) == pytest.approx(40.0, abs=1e-12) and abs(O.silu(-40.0)) < 1e-15


def test_l2norm_unit_norm_and_scale_invariance():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 8))
    n = O.l2norm(x, eps=0.0)
    assert np.allclose(np.linalg.norm(n, axis=-1), 1.0, atol=1e-14)
    assert np.allclose(O.l2norm(7.5 * x, eps=0.0), n, atol=1e-14)
    assert np.array_equal(O.l2norm(np.zeros(8)), np.zeros(8))       # eps keeps zero finite


def test_gates_from_logits_values():
    g, b = O.gates_from_logits(np.array([0.0, 60.0, -60.0]), np.array([0.0, 60.0, -60.0]), -5.0)
    assert g[0] == -2.5 and b[0] == 0.5
    assert g[1] == pytest.approx(-5.0, abs=1e-20) and b[1] == pytest.approx(1.0, abs=1e-20)
    assert g[2] == pytest.approx(0.0, abs=1e-20) and b[2] == pytest.approx(0.0, abs=1e-20)
    a = np.linspace(-6, 6, 101)
    gg, bb = O.gates_from_logits(a, a, -5.0)
    assert np.all(np.diff(gg) < 0) and np.all(np.diff(bb) > 0)      # monotone, opposite ways
    assert gg.min() >= -5.0 and gg.max() <= 0.0 and bb.min() >= 0.0 and bb.max() <= 1.0


def test_input_prep_channel_layout_by_hand():
    """With only the newest tap and no activation the prologue reduces to slicing
    mixed_qkv rows as [q | k | v] per head and normalising q and k per head."""
    H, dk, dv, T = 2, 4, 3, 5
    p = _prologue(T, H, dk, dv, w=3, seed=9)
    C = H * (2 * dk + dv)
    W = np.zeros((C, 3)); W[:, 2] = 1.0
    q, k, v, g, b, _ = O.input_prep(p["mixed"], W, p["window"][0], p["g_logits"], p["beta_logits"],
                                    H, dk, dv, -5.0, act=O.ACT_NONE, eps=0.0)
    x = p["mixed"]
    for t in range(T):
        for h in range(H):
            xq = x[t, h * dk:(h + 1) * dk]
            xk = x[t, H * dk + h * dk:H * dk + (h + 1) * dk]
            assert np.allclose(q[t, h], xq / math.sqrt(sum(c * c for c in xq)), atol=1e-14)
            assert np.allclose(k[t, h], xk / math.sqrt(sum(c * c for c in xk)), atol=1e-14)
            assert np.array_equal(v[t, h], x[t, 2 * H * dk + h * dv:2 * H * dk + (h + 1) * dv])


@pytest.mark.parametrize("act", [0, 1])
def test_input_prep_split_equals_one_shot(act):
    """Carrying the conv window across a cut gives the same values as one pass."""
    H, dk, dv, T = 2, 4, 3, 13
    p = _prologue(T, H, dk, dv, w=4, seed=11)
    args = (H, dk, dv, -5.0, act)
    whole = O.input_prep(p["mixed"], p["weight"], p["window"][0], p["g_logits"], p["beta_logits"], *args)
    a = O.input_prep(p["mixed"][:6], p["weight"], p["window"][0], p["g_logits"][:6], p["beta_logits"][:6], *args)
    b = O.input_prep(p["mixed"][6:], p["weight"], a[5], p["g_logits"][6:], p["beta_logits"][6:], *args)
    for i in range(5):
        assert np.array_equal(np.concatenate([a[i], b[i]]), whole[i])
    assert np.array_equal(b[5], whole[5])
    # the conv checkpoint at a boundary is the window a pass up to it leaves behind
    assert np.array_equal(O.conv_window_at(p["mixed"], p["window"][0], 6), a[5])
    assert np.array_equal(O.conv_window_at(p["mixed"], p["window"][0], T), whole[5])


# --------------------------------------------------------------------------
# Sequence-parallel (segment scan) form
# --------------------------------------------------------------------------
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("seg_len", [1, 3, 7, 40])
def test_segment_scan_equals_recurrent(mode, seg_len):
    """Starts from the affine scan, outputs from each segment's start: the full recurrence."""
    S0, a = _rand_head(23, 5, 4, seed=seg_len + 10 * mode)
    o_ref, S_ref = O.kda_recurrent(S0, a["q"], a["k"], a["v"], a["g"], a["beta"], mode)
    o, S = O.prefill_segment_scan(S0, a["q"], a["k"], a["v"], a["g"], a["beta"], seg_len, mode)
    assert np.abs(o - o_ref).max() < 1e-12 and np.abs(S - S_ref).max() < 1e-12


def test_segment_transition_is_the_homogeneous_recurrence():
    """M applied to a state equals the recurrence run with v = 0 from that state."""
    S0, a = _rand_head(9, 4, 6, seed=77)
    M = O.segment_transition(a["k"], a["g"], a["beta"])
    _, S_h = O.kda_recurrent(S0, a["q"], a["k"], np.zeros_like(a["v"]), a["g"], a["beta"])
    assert np.abs(M @ S0 - S_h).max() < 1e-13
