"""Seeded synthetic input generators: shapes, tree structure, paths, rounding, determinism."""

import numpy as np
import pytest
import torch

from gated_deltanet_tree_03_b300 import workloads as W


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, -1.0, 1e-30, 3.3895e38, 1.00390625, 1.01171875],
                                 np.float32)])
    bits = W.f32_to_bf16_bits(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, want)
    back = W.bf16_bits_to_f32(bits)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("n,F,D", [(16, 4, 8), (64, 4, 8), (32, 3, 6), (40, 1, 63), (7, 2, 2)])
def test_random_tree_limits(n, F, D):
    rng = np.random.default_rng(n * 100 + F)
    for _ in range(20):
        p = W.random_tree_parents(rng, n, fanout_max=F, depth_max=D)
        assert len(p) == n and p[0] == -1
        assert all(-1 <= p[t] < t for t in range(n))
        assert np.sum(p == -1) == 1
        counts = np.bincount(p[p >= 0], minlength=n)
        assert counts.max() <= F
        depth = np.zeros(n, int)
        for t in range(1, n):
            depth[t] = depth[p[t]] + 1
        assert depth.max() <= D


def test_topological_relabel_is_valid():
    rng = np.random.default_rng(3)
    p = W.random_tree_parents(rng, 30, 3, 6)
    for _ in range(10):
        q, perm = W.random_topological_relabel(rng, p)
        assert sorted(perm.tolist()) == list(range(30))
        assert all(-1 <= q[t] < t for t in range(30))
        for t in range(30):  # same edges
            want = p[perm[t]]
            assert (q[t] == -1) == (want == -1)
            if want >= 0:
                assert perm[q[t]] == want


def _check_paths(tb):
    for r in range(tb.B):
        par = tb.request_parent(r)
        L = tb.path_len[r]
        prev = -1
        for i in range(L):
            x = tb.path[r, i]
            assert 0 <= x < len(par) and par[x] == prev
            prev = x
        assert np.all(tb.path[r, L:] == -1)


@pytest.mark.parametrize("idx,batch", [(0, 1), (1, 256), (2, 1), (2, 64), (3, 128), (4, 8)])
def test_config_structure(idx, batch):
    tb = W.make_config(idx, batch=batch, heads=2 if idx else None)
    assert tb.B == batch
    _check_paths(tb)
    sizes = np.diff(tb.cu_nodes)
    if idx == 0:
        assert tb.dk == tb.dv == 32 and tb.H == 1
        assert tb.parent.tolist() == [-1, 0, 1] and tb.path[0, :2].tolist() == [0, 1]
    if idx == 1:
        assert np.all(sizes == 4) and tb.dk == 128
        for r in range(batch):
            assert tb.path[r, :tb.path_len[r]].tolist() == list(range(tb.path_len[r]))
            assert 1 <= tb.path_len[r] <= 4
    if idx == 2:
        assert np.all(sizes == 6)
        assert tb.request_parent(0).tolist() == [-1, 0, 0, 0, 1, 2]
        assert np.all(tb.path_len >= 1)
    if idx == 3:
        assert sizes.min() >= 16 and sizes.max() <= 64 and len(set(sizes.tolist())) > 1
    if idx == 4:
        assert np.all(sizes == 32)
        a = np.exp(tb.g.astype(np.float64))
        assert a.min() >= 0.85 - 1e-6 and a.max() <= 1.0
    # value recipe
    qf = tb.q_f32()
    norms = np.linalg.norm(qf.astype(np.float64), axis=-1)
    assert np.all(np.abs(norms - 1) < 1e-2)
    assert np.all(tb.beta >= 0) and np.all(tb.beta <= 1)
    assert np.all(tb.g <= 0)


def test_config_seeded_and_deterministic():
    a = W.make_config(3, heads=2)
    b = W.make_config(3, heads=2)
    np.testing.assert_array_equal(a.parent, b.parent)
    np.testing.assert_array_equal(a.ST0, b.ST0)
    np.testing.assert_array_equal(a.q, b.q)
    c = W.make_config(4, batch=8, layer=1, heads=2)
    d = W.make_config(4, batch=8, layer=2, heads=2)
    assert not np.array_equal(c.ST0, d.ST0)


def test_state_distribution():
    tb = W.make_config(1, batch=8)
    s = tb.ST0.astype(np.float64)
    assert abs(s.std() - 0.1) < 0.005 and abs(s.mean()) < 0.005
