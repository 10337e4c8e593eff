"""Pins for the draft-budget oracle (``oracle.budget``).

* top-B allocation: the page's own example of the rule (a late position of a confident request
  outranks the first position of an unconfident one), a hand-worked case, and brute force over
  every allocation of B positions as prefixes of the requests' drafts: the top-B pick is the one
  that maximises the expected number of accepted drafts (the sum of the chosen survival
  probabilities, by linearity of expectation), uniquely so when survivals are distinct;
* survival products: closed form on constant probabilities, invalid probabilities count as 0;
* best-first growth: a hand-worked tree, threshold ties (a candidate exactly at the threshold is
  taken; equal values go to the smaller index), and against the reformulation "every candidate
  whose branch value reaches the threshold, sorted by (value desc, index asc), cut at max_nodes",
  which equals the best-first pop order because branch values never grow along a branch;
  ancestor-closed output in parent-before-child order; growth is monotone in the threshold.
"""

import itertools

import numpy as np
import pytest

from oracle import budget as OB


def test_page_example_confident_late_position_beats_unconfident_first():
    p = np.array([[0.95, 0.95, 0.95], [0.6, 0.5, 0.5]], np.float32)
    n, s, cu, parent = OB.topb(p, 3)
    assert s[0, 2] > s[1, 0]  # 0.857 > 0.6
    assert n.tolist() == [3, 0]
    n4, *_ = OB.topb(p, 4)
    assert n4.tolist() == [3, 1]
    assert cu.tolist() == [0, 4, 5]
    assert parent.tolist() == [-1, 0, 1, 2, -1]  # chains: the produced token, then the drafts


def test_survival_closed_form_and_invalid_probabilities():
    p = np.full((2, 5), 0.5, np.float32)
    s = OB.survival(p)
    np.testing.assert_array_equal(s[0], np.float32(0.5) ** np.arange(1, 6, dtype=np.float32))
    bad = np.array([[0.9, np.nan, 0.9], [0.9, 1.5, 0.9], [-0.1, 0.9, 0.9]], np.float32)
    sb = OB.survival(bad)
    assert sb[0, 0] == np.float32(0.9) and sb[0, 1] == 0 and sb[0, 2] == 0
    assert sb[1, 1] == 0 and sb[2, 0] == 0


def _best_prefix_allocation(s, B):
    R, K = s.shape
    best, arg = -1.0, None
    for alloc in itertools.product(range(K + 1), repeat=R):
        if sum(alloc) != B:
            continue
        v = sum(float(np.sum(s[r, :alloc[r]], dtype=np.float64)) for r in range(R))
        if v > best + 1e-12:
            best, arg = v, alloc
    return list(arg)


@pytest.mark.parametrize("seed", range(6))
def test_topb_maximises_expected_accepted_drafts(seed):
    rng = np.random.default_rng(seed)
    R, K = 3, 4
    p = rng.uniform(0.2, 1.0, size=(R, K)).astype(np.float32)
    s = OB.survival(p)
    for B in range(0, R * K + 1):
        n, *_ = OB.topb(p, B)
        assert n.tolist() == _best_prefix_allocation(s, B), B


@pytest.mark.parametrize("seed", range(4))
def test_topb_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    R, K = 37, 7
    conf = rng.uniform(0.3, 0.97, size=(R, 1))
    p = np.clip(conf + rng.normal(0, 0.05, size=(R, K)), 0, 1).astype(np.float32)
    for B in (0, 1, 50, R * K - 1, R * K, R * K + 9):
        n, s, cu, parent = OB.topb(p, B)
        assert n.sum() == min(B, R * K)
        chosen = np.zeros((R, K), bool)
        for r in range(R):
            chosen[r, :n[r]] = True
        if chosen.any() and (~chosen).any():
            assert s[chosen].min() >= s[~chosen].max()
        assert cu[-1] == R + n.sum() and len(parent) == cu[-1]
        for r in range(R):
            assert parent[cu[r]:cu[r + 1]].tolist() == list(range(-1, n[r]))


def test_growth_hand_example():
    # complete binary candidate tree of depth 2: 0 -> (1, 2), 1 -> (3, 4), 2 -> (5, 6)
    p = np.array([[0.0, 0.8, 0.3, 0.5, 0.6, 0.9, 0.2]], np.float32)
    out = OB.grow_best_first(p, 2, 2, 0.35, 10)
    # values: 1: 0.8, 4: 0.48, 3: 0.4, 2: 0.3 (< 0.35, growth stops)
    assert out["n_nodes"].tolist() == [4]
    assert out["cand"][0, :4].tolist() == [0, 1, 4, 3]
    assert out["parent_local"][0, :4].tolist() == [-1, 0, 1, 1]
    np.testing.assert_allclose(out["value"][0, :4], [1.0, 0.8, 0.48, 0.4], rtol=1e-6)
    assert out["cu_nodes"].tolist() == [0, 4] and out["parent"].tolist() == [-1, 0, 1, 1]
    cap = OB.grow_best_first(p, 2, 2, 0.35, 2)
    assert cap["cand"][0].tolist() == [0, 1]


def test_growth_threshold_ties_and_degenerate_limits():
    p = np.array([[0.0, 0.5, 0.5]], np.float32)
    out = OB.grow_best_first(p, 2, 1, 0.5, 8)
    assert out["cand"][0, :3].tolist() == [0, 1, 2]  # at the threshold is taken; tie -> smaller index
    assert OB.grow_best_first(p, 2, 1, 0.5000001, 8)["n_nodes"].tolist() == [1]
    assert OB.grow_best_first(p, 2, 1, 2.0, 8)["n_nodes"].tolist() == [1]  # the root is always taken
    assert OB.grow_best_first(p, 2, 1, 0.0, 1)["n_nodes"].tolist() == [1]
    assert OB.grow_best_first(p, 2, 1, 0.0, 0)["n_nodes"].tolist() == [0]


def _sorted_reformulation(p, fanout, depth, thr, max_nodes):
    C = p.shape[0]
    v = np.zeros(C, np.float32)
    v[0] = 1
    for c in range(1, C):
        v[c] = np.float32(v[(c - 1) // fanout] * OB._prob(p[c]))
    keep = [c for c in range(C) if c == 0 or v[c] >= np.float32(thr)]
    keep.sort(key=lambda c: (-float(v[c]), c))
    return keep[:max_nodes]


@pytest.mark.parametrize("fanout,depth,thr,max_nodes", [(2, 5, 0.05, 64), (3, 4, 0.02, 32), (4, 3, 0.1, 64),
                                                      (1, 9, 0.3, 64), (3, 5, 0.0, 64)])
def test_growth_equals_sorted_reformulation(fanout, depth, thr, max_nodes):
    rng = np.random.default_rng(fanout * 10 + depth)
    C = OB.candidate_count(fanout, depth)
    R = 9
    p = rng.dirichlet(np.full(fanout + 1, 0.5), size=(R, C)).astype(np.float32)[:, :, 0]
    p[:, ::5] = 0.5  # some exactly repeated values to exercise ties
    out = OB.grow_best_first(p, fanout, depth, thr, max_nodes)
    for r in range(R):
        n = int(out["n_nodes"][r])
        cand = out["cand"][r, :n].tolist()
        assert cand == _sorted_reformulation(p[r], fanout, depth, thr, max_nodes)
        par = out["parent_local"][r, :n]
        assert all(par[t] < t for t in range(n))  # parent before child
        idx = {c: t for t, c in enumerate(cand)}
        assert all(par[t] == (-1 if c == 0 else idx[(c - 1) // fanout]) for t, c in enumerate(cand))
        assert np.all(np.diff(out["value"][r, :n]) <= 0)


def test_growth_is_monotone_in_threshold():
    rng = np.random.default_rng(7)
    C = OB.candidate_count(3, 4)
    p = rng.uniform(0, 1, size=(4, C)).astype(np.float32)
    prev = None
    for thr in (0.5, 0.2, 0.1, 0.05, 0.01):
        out = OB.grow_best_first(p, 3, 4, thr, 200)
        sets = [set(out["cand"][r, :out["n_nodes"][r]].tolist()) for r in range(4)]
        if prev is not None:
            assert all(a <= b for a, b in zip(prev, sets))
        prev = sets
