"""Planted mistakes in the oracles of the serving layouts, the draft budgeting and tree attention.

Each mutation is a plausible slip in one of those oracles: a wrong head mapping, a lost sign, a
missed scale, an ignored slot, a sum for a product, a reversed order, a strict threshold, a
dropped cap, a NaN counted as certain, the node itself not visible, or every earlier index
visible. It is planted with monkeypatch, and at least one of that oracle's pins must then fail.
"""

import numpy as np
import pytest

from oracle import attention as OA
from oracle import budget as OB
from oracle import serving as OS

import test_attention_pins as AP
import test_budget_pins as BP
import test_serving_pins as SP

SERVING_PINS = [
    SP.test_softplus_closed_forms_and_identities,
    SP.test_sigmoid_closed_forms_and_symmetry,
    lambda: SP.test_gate_decay_is_a_power_of_the_logistic(3.0),
    lambda: SP.test_serving_verify_matches_brute_force_replay(4, 2, True),
    lambda: SP.test_serving_verify_matches_brute_force_replay(4, 1, False),
    SP.test_serving_commit_matches_brute_force_and_leaves_other_slots,
    SP.test_pool_permutation_invariance_and_plain_special_case,
    SP.test_output_is_linear_in_the_query_scale,
]

BUDGET_PINS = [
    BP.test_page_example_confident_late_position_beats_unconfident_first,
    BP.test_survival_closed_form_and_invalid_probabilities,
    lambda: BP.test_topb_maximises_expected_accepted_drafts(0),
    lambda: BP.test_topb_invariants(0),
    BP.test_growth_hand_example,
    BP.test_growth_threshold_ties_and_degenerate_limits,
    lambda: BP.test_growth_equals_sorted_reformulation(2, 5, 0.05, 64),
    BP.test_growth_is_monotone_in_threshold,
]

ATTENTION_PINS = [
    lambda: AP.test_matches_library_attention_with_ancestor_mask(1, 4, 2, (0, 40)),
    AP.test_chain_is_causal_attention,
    AP.test_root_without_prefix_returns_its_value_and_equal_keys_average,
    AP.test_branch_extraction_prefix_permutation_and_relabelling,
]


def _failures(pins):
    n = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError, ZeroDivisionError, KeyError):
            n += 1
    return n


def test_unmutated_oracles_pass_every_pin():
    assert _failures(SERVING_PINS + BUDGET_PINS + ATTENTION_PINS) == 0


# ------------------------------------------------------------------ serving layouts
_expand, _gate_beta, _verify, _states = OS.expand_heads, OS.gate_beta, OS.verify, OS._states


def _heads_modulo(x, H):  # value head h reads key head h % H_qk instead of h // (H / H_qk)
    x = np.asarray(x, dtype=np.float64)
    return x[:, np.arange(H) % x.shape[1], :]


def _decay_sign_lost(a_raw, b_raw, A_log, dt_bias):
    g, beta = _gate_beta(a_raw, b_raw, A_log, dt_bias)
    return -g, beta


def _sigmoid_flipped(a_raw, b_raw, A_log, dt_bias):
    g, beta = _gate_beta(a_raw, b_raw, A_log, dt_bias)
    return g, 1.0 - beta


def _softplus_wrong(x):  # ln(1 + x) for ln(1 + e^x)
    return np.log1p(np.abs(np.asarray(x, dtype=np.float64)))


def _scale_ignored(*args, q_scale=1.0, gates=None):
    return _verify(*args, q_scale=1.0, gates=gates)


def _slot_ignored(pool, slot):
    slot = np.asarray(slot)
    live = slot >= 0
    return np.asarray(pool, dtype=np.float64)[np.arange(len(slot)) % len(pool)], live


@pytest.mark.parametrize("name,fn", [("expand_heads", _heads_modulo), ("gate_beta", _decay_sign_lost),
                                     ("gate_beta", _sigmoid_flipped), ("softplus", _softplus_wrong),
                                     ("verify", _scale_ignored), ("_states", _slot_ignored)],
                         ids=["heads_modulo", "decay_sign", "sigmoid_flipped", "softplus", "scale_ignored",
                              "slot_ignored"])
def test_serving_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(OS, name, fn)
    assert _failures(SERVING_PINS) >= 1


# ------------------------------------------------------------------ draft budgeting
_survival, _topb, _grow, _prob = OB.survival, OB.topb, OB.grow_best_first, OB._prob


def _survival_sum(p_accept):  # a running sum for the running product
    p = np.asarray(p_accept, dtype=np.float32)
    return np.cumsum(np.where((p >= 0) & (p <= 1), p, 0), axis=1).astype(np.float32)


def _topb_ascending(p_accept, budget):  # the budget to the smallest survivals
    return _topb(-np.asarray(p_accept, dtype=np.float32) + 1.0, budget)


def _grow_strict(p_edge, fanout, depth, threshold, max_nodes):  # "value > threshold"
    return _grow(p_edge, fanout, depth, float(np.nextafter(np.float32(threshold), np.float32(np.inf))), max_nodes)


def _grow_uncapped(p_edge, fanout, depth, threshold, max_nodes):
    return _grow(p_edge, fanout, depth, threshold, max(max_nodes, 64))


def _prob_nan_is_certain(x):
    x = np.float32(x)
    return np.float32(1) if np.isnan(x) else _prob(x)


@pytest.mark.parametrize("name,fn", [("survival", _survival_sum), ("topb", _topb_ascending),
                                     ("grow_best_first", _grow_strict), ("grow_best_first", _grow_uncapped),
                                     ("_prob", _prob_nan_is_certain)],
                         ids=["sum_for_product", "ascending", "strict_threshold", "uncapped", "nan_certain"])
def test_budget_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(OB, name, fn)
    assert _failures(BUDGET_PINS) >= 1


# ------------------------------------------------------------------ tree attention
_root_path, _attention = OA._root_path, OA.tree_attention


def _self_not_visible(par, t):
    return _root_path(par, t)[:-1]


def _all_earlier_visible(par, t):  # causal over the index order instead of the ancestors
    return list(range(t + 1))


def _attention_scale_ignored(q, k, v, k_cache, v_cache, cu_prefix, parent, cu_nodes, scale):
    return _attention(q, k, v, k_cache, v_cache, cu_prefix, parent, cu_nodes, 1.0)


@pytest.mark.parametrize("name,fn", [("_root_path", _self_not_visible), ("_root_path", _all_earlier_visible),
                                     ("tree_attention", _attention_scale_ignored)],
                         ids=["self_not_visible", "all_earlier_visible", "scale_ignored"])
def test_attention_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(OA, name, fn)
    assert _failures(ATTENTION_PINS) >= 1
