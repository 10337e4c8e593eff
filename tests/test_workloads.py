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


def test_serving_batch_recipe():
    tb, sv = W.make_serving_batch(seed=4, B=9, H=8, H_qk=2, d=16, n_range=(1, 7), n_slots=30, pad_every=4)
    assert sv.pool.shape == (30, 8, 16, 16) and sv.pool.dtype == np.float32
    assert sv.q.shape == (tb.T, 2, 16) and sv.k.shape == (tb.T, 2, 16) and sv.q.dtype == np.uint16
    live = sv.slot[sv.slot >= 0]
    assert len(set(live.tolist())) == len(live) and np.all(live < 30)  # distinct slots inside the pool
    assert sv.slot[3] == -1 and sv.slot[7] == -1 and np.sum(sv.slot == -1) == 2
    assert abs(sv.q_scale - 16 ** -0.5) < 1e-12
    assert np.all(sv.dt_bias >= -7) and np.all(sv.dt_bias <= -2)
    assert np.all(np.exp(sv.A_log) >= 1 - 1e-6) and np.all(np.exp(sv.A_log) <= 16 + 1e-5)
    # L2-normalised keys before bf16 rounding
    k = W.bf16_bits_to_f32(sv.k)
    np.testing.assert_allclose(np.linalg.norm(k, axis=-1), 1.0, atol=2e-2)
    tb2, sv2 = W.make_serving_batch(seed=4, B=9, H=8, H_qk=2, d=16, n_range=(1, 7), n_slots=30, pad_every=4)
    assert np.array_equal(sv.slot, sv2.slot) and np.array_equal(sv.a_raw, sv2.a_raw)
    with pytest.raises(ValueError):
        W.make_serving_batch(seed=4, B=9, H=8, H_qk=2, d=16, n_slots=5)


def test_acceptance_draws_have_the_reported_spread():
    rng = np.random.default_rng(0)
    p = W.draw_acceptance(rng, 4096, 7)
    assert p.dtype == np.float32 and np.all((p >= 0) & (p <= 1))
    s = np.cumprod(p.astype(np.float64), axis=1)
    assert s[:, 0].mean() > 0.7 and s[:, 6].mean() < 0.1  # first of seven drafts > 70 %, last < 10 %


def test_candidate_tree_draws():
    rng = np.random.default_rng(1)
    fanout, depth = 3, 4
    p = W.draw_edge_probs(rng, 5, fanout, depth)
    C = sum(fanout ** l for l in range(depth + 1))
    assert p.shape == (5, C) and np.all(p[:, 0] == 1)
    kids = p[:, 1:].reshape(5, -1, fanout)
    assert np.all(np.diff(kids, axis=2) <= 0)  # siblings sorted, most likely first
    assert np.all(kids.sum(axis=2) <= 1 + 1e-6)  # one Dirichlet draw shared with "none accepted"


def test_attention_batch_layout():
    parents = [W.root_branch_parents(), W.chain_parents(3)]
    ab = W.make_attention_batch(2, B=2, Hq=8, Hkv=2, d=64, prefix_range=(5, 9), parents=parents)
    assert ab.T == 9 and ab.cu_nodes.tolist() == [0, 6, 9]
    assert ab.q.shape == (9, 8, 64) and ab.k.shape == (9, 2, 64) and ab.v.shape == (9, 2, 64)
    assert ab.k_cache.shape == (ab.P, 2, 64) and 10 <= ab.P <= 18
    assert np.all(np.diff(ab.cu_prefix) >= 5) and np.all(np.diff(ab.cu_prefix) <= 9)
    assert abs(ab.scale - 64 ** -0.5) < 1e-12 and ab.max_nodes == 6


@pytest.mark.parametrize("cfg,batch,layer", [(0, 1, 0), (1, 256, 0), (2, 1, 0), (2, 64, 0), (3, 128, 0), (4, 8, 7),
                                             (4, 128, 47)])
def test_config_shape_matches_make_config(cfg, batch, layer):
    """The device-timed presets use the same trees and accepted paths as the host presets."""
    s = W.config_shape(cfg, batch, layer)
    t = W.make_config(cfg, batch=batch, layer=layer)
    for key in ("parent", "cu_nodes", "path", "path_len"):
        np.testing.assert_array_equal(getattr(s, key), getattr(t, key))
    assert (s.B, s.H, s.dk, s.dv, s.T, s.max_nodes, s.max_path) == (t.B, t.H, t.dk, t.dv, t.T, t.max_nodes,
                                                                     t.max_path)


@pytest.mark.parametrize("cfg", [2, 4])
def test_draw_values_device_recipe(cfg):
    """Device-drawn values follow the preset recipe (drawn here on the CPU device)."""
    import torch
    s = W.config_shape(cfg, 64 if cfg == 2 else 32, 0)
    v = W.draw_values_device(s, seed=5, device="cpu")
    T, H = s.T, s.H
    assert v["ST"].shape == (s.B, H, 128, 128) and v["ST"].dtype == torch.float32
    assert abs(float(v["ST"].std()) - 0.1) < 0.005
    for key in ("q", "k"):
        assert v[key].shape == (T, H, 128) and v[key].dtype == torch.bfloat16
        norms = v[key].float().norm(dim=-1)
        assert float((norms - 1).abs().max()) < 0.02
    assert v["v"].dtype == torch.bfloat16 and abs(float(v["v"].float().std()) - 1) < 0.05
    assert float(v["beta"].min()) >= 0 and float(v["beta"].max()) <= 1
    a = torch.exp(v["g"])
    if cfg == 4:
        assert float(a.min()) >= 0.85 - 1e-6 and float(a.max()) <= 1.0
    else:
        assert float(v["g"].max()) <= 0 and abs(float(v["g"].mean()) + 0.1 * 0.8) < 0.02  # E softplus(N(0,1)) ~ 0.806
    again = W.draw_values_device(s, seed=5, device="cpu")
    assert torch.equal(again["q"], v["q"])
    np.testing.assert_array_equal(v["parent"].numpy(), s.parent)
