"""Pins for the greedy-acceptance oracle: hand-worked trees and the properties that define the
rule (a root-to-node chain, every step a match, no matching child left at the end, the lowest
index among matching siblings, truncation at max_path)."""

import numpy as np
import pytest

import oracle
from gated_deltanet_tree_03_b300 import workloads as W


def _one(parent, draft, target, max_path=8):
    cu = np.array([0, len(parent)], np.int32)
    path, plen, trunc = oracle.accept_greedy(np.asarray(draft), np.asarray(target), np.asarray(parent, np.int32), cu,
                                             max_path)
    return list(path[0, :plen[0]]), bool(trunc[0])


def test_hand_worked_chain_and_branches():
    # chain 0-1-2-3: target after 0 is 7 (= draft of 1), after 1 is 9 (= draft of 2), after 2 is 4 (!= 5)
    assert _one([-1, 0, 1, 2], [0, 7, 9, 5], [7, 9, 4, 0]) == ([0, 1, 2], False)
    # root with children 1, 2, 3 (drafts 5, 6, 6); target after 0 is 6 -> the lowest index 2
    # then node 2 has child 4 (draft 8); target after 2 is 8 -> 4
    assert _one([-1, 0, 0, 0, 2], [0, 5, 6, 6, 8], [6, 0, 8, 0, 0]) == ([0, 2, 4], False)
    # nothing matches: only the root
    assert _one([-1, 0, 0], [0, 1, 2], [3, 0, 0]) == ([0], False)
    # truncation
    assert _one([-1, 0, 1, 2], [0, 1, 2, 3], [1, 2, 3, 0], max_path=2) == ([0, 1], True)
    # a later root is never entered
    assert _one([-1, -1, 1], [0, 4, 5], [4, 5, 0]) == ([0], False)


def test_rule_properties_on_random_trees():
    rng = np.random.default_rng(3)
    for trial in range(40):
        tb = W.make_random_batch(seed=200 + trial, B=4, H=1, d=8, n_range=(1, 40), fanout_max=4, depth_max=8)
        draft, target = W.draw_tokens(rng, tb.parent, tb.cu_nodes, vocab=6, p_match=0.8)
        path, plen, trunc = oracle.accept_greedy(draft, target, tb.parent, tb.cu_nodes, 64)
        for r in range(tb.B):
            t0, n = tb.cu_nodes[r], tb.n_nodes(r)
            L = plen[r]
            if n == 0:
                assert L == 0
                continue
            seq = list(path[r, :L])
            assert seq[0] == 0 and np.all(path[r, L:] == -1) and not trunc[r]
            for a, b in zip(seq, seq[1:]):
                assert tb.parent[t0 + b] == a and draft[t0 + b] == target[t0 + a]
                lower = [c for c in range(a + 1, b) if tb.parent[t0 + c] == a and draft[t0 + c] == target[t0 + a]]
                assert not lower  # the lowest-indexed matching child was taken
            last = seq[-1]
            assert not [c for c in range(n) if tb.parent[t0 + c] == last and draft[t0 + c] == target[t0 + last]]


def test_malformed_tree_rejected():
    with pytest.raises(ValueError):
        _one([-1, 1, 0], [0, 0, 0], [0, 0, 0])
