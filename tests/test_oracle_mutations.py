"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Each mutant is the oracle's own source with one expression changed, compiled
into the oracle module's namespace and patched in for the duration of a test.
A mutant that no pin catches would mean the pins leave that part of the
oracle unchecked.
"""
import inspect
import textwrap

import numpy as np
import pytest
import torch

from oracle import kda_oracle as O
from kda_delta_rule_gb300 import inputs as I

import test_oracle_pins as pins


def _mutant(fn, old, new):
    src = textwrap.dedent(inspect.getsource(fn))
    assert src.count(old) >= 1, (fn.__name__, old)
    src = src.replace(old, new, 1)
    ns = dict(vars(O))
    exec(compile(src, f"<mutant {fn.__name__}>", "exec"), ns)
    return ns[fn.__name__]


STEP_MUTANTS = {
    "decay_first_uses_undecayed_delta": (
        'delta = v - np.einsum("...ij,...i->...j", S_dec, k)',
        'delta = v - np.einsum("...ij,...i->...j", S, k)'),
    "update_sign_flipped": (
        "S_new = S_dec + b * k[..., :, None] * delta[..., None, :]",
        "S_new = S_dec - b * k[..., :, None] * delta[..., None, :]"),
    "beta_dropped": (
        "S_new = S_dec + b * k[..., :, None] * delta[..., None, :]",
        "S_new = S_dec + k[..., :, None] * delta[..., None, :]"),
    "decay_on_value_axis": (
        "decay = np.exp(g)[..., :, None]",
        "decay = np.exp(g)[..., None, :1]"),
    "readout_before_write": (
        'o = np.einsum("...ij,...i->...j", S_new, q)',
        'o = np.einsum("...ij,...i->...j", S, q)'),
    "readout_transposed": (
        'o = np.einsum("...ij,...i->...j", S_new, q)',
        'o = np.einsum("...ij,...j->...i", S_new, q)'),
    "page1_decays_before_delta": (
        'delta = v - np.einsum("...ij,...i->...j", S, k)\n        S_new = decay * S',
        'delta = v - np.einsum("...ij,...i->...j", decay * S, k)\n        S_new = decay * S'),
}

CHUNK_MUTANTS = {
    "P_mask_drops_diagonal": ("EP = np.exp(np.where(lower[:, :, None]",
                              "EP = np.exp(np.where(lower_strict[:, :, None]"),
    "A_without_beta": ('A = np.einsum("ri,si,rsi->rs", k, k, EA) * beta[None, :]',
                       'A = np.einsum("ri,si,rsi->rs", k, k, EA)'),
    "page1_shift_missing": ("G = Gam if mode == DECAY_FIRST else Gam - g", "G = Gam"),
    "output_uses_unscaled_delta": ("O = (q * np.exp(Gam)) @ S + P @ bD",
                                   "O = (q * np.exp(Gam)) @ S + P @ Delta"),
    "state_decay_missing": ("S_end = np.exp(GL)[:, None] * S +", "S_end = S +"),
    "wy_sign": ("Delta = U - W @ S", "Delta = U + W @ S"),
}


def _step_pins():
    for mode in (O.DECAY_FIRST, O.UNDECAYED_DELTA):
        for T, dk, dv, seed in [(2, 4, 3, 1), (3, 5, 5, 2)]:
            yield lambda m=mode, a=(T, dk, dv, seed): pins.test_recurrent_equals_unrolled_products(m, *a)
    yield pins.test_scalar_step_by_hand
    yield pins.test_two_by_two_step_by_hand
    yield pins.test_decay_first_perfect_write_and_page1_breaks_it
    yield pins.test_cold_start_single_token


def _caught(pin_iter):
    for pin in pin_iter:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            return True
    return False


@pytest.mark.parametrize("name", sorted(STEP_MUTANTS))
def test_step_mutant_is_caught(name, monkeypatch):
    old, new = STEP_MUTANTS[name]
    monkeypatch.setattr(O, "kda_step", _mutant(O.kda_step, old, new))
    assert _caught(_step_pins()), f"no pin catches mutant {name}"


@pytest.mark.parametrize("name", sorted(CHUNK_MUTANTS))
def test_chunk_mutant_is_caught(name, monkeypatch):
    old, new = CHUNK_MUTANTS[name]
    monkeypatch.setattr(O, "chunk_step", _mutant(O.chunk_step, old, new))
    checks = [lambda m=m: pins.test_chunked_equals_recurrent(m, 200, 64)
              for m in (O.DECAY_FIRST, O.UNDECAYED_DELTA)]
    assert _caught(checks), f"no pin catches mutant {name}"


def test_unmutated_oracle_passes_the_same_pins():
    assert not _caught(_step_pins())


RING_MUTANTS = {
    "ring_drops_newest": ("self._steps.pop(0)", "self._steps.pop()"),
    "ring_grows_past_capacity": ("if len(self._steps) == self.capacity:",
                                 "if len(self._steps) > self.capacity:"),
}


@pytest.mark.parametrize("name", sorted(RING_MUTANTS))
def test_ring_mutant_is_caught(name, monkeypatch):
    old, new = RING_MUTANTS[name]
    monkeypatch.setattr(O.RawInputRing, "push", _mutant(O.RawInputRing.push, old, new))
    checks = [pins.test_ring_window_sizes_printed, pins.test_ring_overwrites_oldest_first,
              lambda: pins.test_ring_replay_equals_recurrent(0)]
    assert _caught(checks), f"no pin catches mutant {name}"


PROLOGUE_MUTANTS = {
    "conv_taps_reversed": ("short_conv", "y[t] += weight[:, j] * z[t + j]", "y[t] += weight[:, w - 1 - j] * z[t + j]"),
    "conv_window_dropped": ("short_conv", "z = np.concatenate([_f64(window), x], axis=0)",
                            "z = np.concatenate([0.0 * _f64(window), x], axis=0)"),
    "conv_window_out_stale": ("short_conv", "return y, z[T:].copy()", "return y, z[:w - 1].copy()"),
    "l2norm_wrong_axis": ("l2norm", "axis=-1", "axis=0"),
    "gate_sign_flipped": ("gates_from_logits", "g_min * sigmoid(g_logits)", "g_min * sigmoid(-g_logits)"),
    "silu_without_x": ("silu", "return x * sigmoid(x)", "return sigmoid(x)"),
    "q_reads_k_columns": ("input_prep", "q = l2norm(y[:, :H * dk]", "q = l2norm(y[:, H * dk:2 * H * dk]"),
}


@pytest.mark.parametrize("name", sorted(PROLOGUE_MUTANTS))
def test_prologue_mutant_is_caught(name, monkeypatch):
    fn, old, new = PROLOGUE_MUTANTS[name]
    monkeypatch.setattr(O, fn, _mutant(getattr(O, fn), old, new))
    checks = [lambda: pins.test_short_conv_is_numpy_correlation(4), pins.test_short_conv_newest_and_oldest_taps,
              pins.test_activation_and_sigmoid_closed_forms, pins.test_l2norm_unit_norm_and_scale_invariance,
              pins.test_gates_from_logits_values, pins.test_input_prep_channel_layout_by_hand,
              lambda: pins.test_input_prep_split_equals_one_shot(1)]
    assert _caught(checks), f"no pin catches mutant {name}"


def test_prologue_pins_pass_unmutated():
    pins.test_short_conv_is_numpy_correlation(4)
    pins.test_short_conv_newest_and_oldest_taps()
    pins.test_input_prep_channel_layout_by_hand()
    pins.test_input_prep_split_equals_one_shot(1)


SCAN_MUTANTS = {
    "transition_product_reversed": ("segment_transition", "M = transition_matrix(k[t], g[t], beta[t], mode) @ M",
                                    "M = M @ transition_matrix(k[t], g[t], beta[t], mode)"),
    "local_state_from_start": ("prefill_segment_scan", "kda_recurrent(np.zeros_like(X),", "kda_recurrent(X,"),
}


@pytest.mark.parametrize("name", sorted(SCAN_MUTANTS))
def test_scan_mutant_is_caught(name, monkeypatch):
    fn, old, new = SCAN_MUTANTS[name]
    monkeypatch.setattr(O, fn, _mutant(getattr(O, fn), old, new))
    checks = [lambda: pins.test_segment_scan_equals_recurrent(0, 7),
              pins.test_segment_transition_is_the_homogeneous_recurrence]
    assert _caught(checks), f"no pin catches mutant {name}"


BOOKKEEPING_MUTANTS = {
    "pack_transposes_heads": ("pack_heads", "np.ascontiguousarray(S).reshape(-1)",
                              "np.ascontiguousarray(np.swapaxes(S, -1, -2)).reshape(-1)"),
    "unpack_reads_value_major": ("unpack_heads", ".reshape(B, H, dk, dv)", ".reshape(B, H, dv, dk).swapaxes(-1, -2)"),
    "page_tail_not_zeroed": ("store_kda", "page = np.zeros(page_elems, dtype=flat.dtype)",
                             "page = np.ones(page_elems, dtype=flat.dtype)"),
    "checkpoint_includes_start": ("checkpoint_positions", "range(1, int(L) // int(ckpt_stride) + 1)",
                                  "range(0, int(L) // int(ckpt_stride) + 1)"),
    "checkpoint_drops_end": ("checkpoint_positions", "range(1, int(L) // int(ckpt_stride) + 1)",
                             "range(1, int(L) // int(ckpt_stride))"),
    "chunked_checkpoint_before_chunk": ("prefill_chunked", "ckpts.append((n, pos, S.copy()))",
                                        "ckpts.append((n, pos - L, S.copy()))"),
    "replay_count_not_clamped": ("verify_and_replay_batched", "n_b = int(min(max(int(n_accepted[b]), 0), draft))",
                                 "n_b = int(n_accepted[b])"),
    "ratio_counts_two_key_vectors": ("snapshot_cost_ratio", "(3 * dk + dv + 1)", "(2 * dk + dv + 1)"),
    "ratio_drops_beta": ("snapshot_cost_ratio", "(3 * dk + dv + 1)", "(3 * dk + dv)"),
}


@pytest.mark.parametrize("name", sorted(BOOKKEEPING_MUTANTS))
def test_bookkeeping_mutant_is_caught(name, monkeypatch):
    fn, old, new = BOOKKEEPING_MUTANTS[name]
    monkeypatch.setattr(O, fn, _mutant(getattr(O, fn), old, new))
    checks = [pins.test_pack_layout_and_roundtrip, pins.test_store_load_zero_padded_page,
              pins.test_checkpoint_positions_long_prefill, pins.test_last_checkpoint_is_final_state_bitwise,
              pins.test_batched_replay_zero_pads_and_matches_per_sequence,
              pins.test_replay_counts_clamp_to_the_draft,
              pins.test_snapshot_cost_ratio_printed_values, pins.test_snapshot_cost_ratio_properties,
              pins.test_varlen_is_independent_sequences]
    assert _caught(checks), f"no pin catches mutant {name}"


def test_bookkeeping_pins_pass_unmutated():
    assert not _caught([pins.test_pack_layout_and_roundtrip, pins.test_store_load_zero_padded_page,
                        pins.test_checkpoint_positions_long_prefill, pins.test_last_checkpoint_is_final_state_bitwise,
                        pins.test_batched_replay_zero_pads_and_matches_per_sequence,
                        pins.test_replay_counts_clamp_to_the_draft,
                        pins.test_snapshot_cost_ratio_printed_values, pins.test_snapshot_cost_ratio_properties,
                        pins.test_varlen_is_independent_sequences])


FORM_MUTANTS = {
    "ut_inverse_sign": ("ut_inverse", "T[r] -= A[r, s] * T[s]", "T[r] += A[r, s] * T[s]"),
    "ut_inverse_transposed": ("ut_inverse", "T[r] -= A[r, s] * T[s]", "T[r] -= A[s, r] * T[s]"),
    "transition_decay_applied_after": ("transition_matrix", "return (np.eye(k.shape[0]) - kkT) @ D",
                                       "return D @ (np.eye(k.shape[0]) - kkT)"),
    "transition_page1_as_decay_first": ("transition_matrix", "return D - kkT", "return (np.eye(k.shape[0]) - kkT) @ D"),
    "conv_window_one_late": ("conv_window_at", "z[boundary:boundary + wm1]", "z[boundary + 1:boundary + 1 + wm1]"),
    "recurrent_checkpoint_one_early": ("prefill_recurrent", "(t + 1 - a) % ckpt_stride == 0", "(t - a) % ckpt_stride == 0"),
}


def _form_pins():
    yield lambda: pins.test_ut_inverse_is_the_inverse()
    for mode in (O.DECAY_FIRST, O.UNDECAYED_DELTA):
        for a in [(2, 4, 3, 1), (3, 5, 5, 2)]:
            yield lambda m=mode, a=a: pins.test_recurrent_equals_unrolled_products(m, *a)
        yield lambda m=mode: pins.test_chunked_equals_recurrent(m, 200, 64)
    yield pins.test_checkpoint_positions_long_prefill
    yield pins.test_last_checkpoint_is_final_state_bitwise
    yield lambda: pins.test_input_prep_split_equals_one_shot(1)
    yield pins.test_input_prep_channel_layout_by_hand


@pytest.mark.parametrize("name", sorted(FORM_MUTANTS))
def test_form_mutant_is_caught(name, monkeypatch):
    fn, old, new = FORM_MUTANTS[name]
    monkeypatch.setattr(O, fn, _mutant(getattr(O, fn), old, new))
    assert _caught(_form_pins()), f"no pin catches mutant {name}"


def test_form_pins_pass_unmutated():
    assert not _caught(_form_pins())
