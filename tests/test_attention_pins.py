"""Pins for the tree-bias attention oracle (``oracle.attention``).

* against PyTorch's scaled_dot_product_attention (a library routine, fp64 on the CPU) with an
  explicit boolean mask - prefix visible, draft node j visible to node t iff j is on t's
  root-to-node path - and, for chains, with the library's own causal mask;
* closed forms: a root node with no prefix sees only itself (o = v); identical keys, or a zero
  scale, give the plain mean of the visible values;
* invariants: branch extraction (a node's output equals that of its root-to-node path verified
  as a chain), permuting the prefix changes nothing, relabelling the tree in another
  topological order permutes the outputs, grouped heads read their own key/value head.
"""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from gated_deltanet_tree_03_b300 import workloads as W


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _args(ab):
    return (_f64(ab.q), _f64(ab.k), _f64(ab.v), _f64(ab.k_cache), _f64(ab.v_cache), ab.cu_prefix, ab.parent,
            ab.cu_nodes, ab.scale)


def _sdpa(ab, causal_chain=False):
    """Library attention per (request, head) with the visibility mask written as a boolean matrix."""
    q, k, v, kc, vc = (_f64(x) for x in (ab.q, ab.k, ab.v, ab.k_cache, ab.v_cache))
    G = ab.Hq // ab.Hkv
    out = np.zeros_like(q)
    for r in range(ab.B):
        t0, t1 = ab.cu_nodes[r], ab.cu_nodes[r + 1]
        p0, p1 = ab.cu_prefix[r], ab.cu_prefix[r + 1]
        n, P = t1 - t0, p1 - p0
        par = ab.parent[t0:t1]
        vis = np.zeros((n, n), bool)
        for t in range(n):
            x = t
            while x >= 0:
                vis[t, x] = True
                x = par[x]
        for h in range(ab.Hq):
            g = h // G
            Q = torch.from_numpy(q[t0:t1, h][None])
            K = torch.from_numpy(np.concatenate([kc[p0:p1, g], k[t0:t1, g]])[None])
            V = torch.from_numpy(np.concatenate([vc[p0:p1, g], v[t0:t1, g]])[None])
            if causal_chain and P == 0:
                o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=ab.scale)
            else:
                mask = torch.from_numpy(np.concatenate([np.ones((n, P), bool), vis], axis=1)[None])
                o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=ab.scale)
            out[t0:t1, h] = o[0].numpy()
    return out


@pytest.mark.parametrize("seed,Hq,Hkv,prefix", [(1, 4, 2, (0, 40)), (2, 8, 1, (5, 60)), (3, 2, 2, (0, 0))])
def test_matches_library_attention_with_ancestor_mask(seed, Hq, Hkv, prefix):
    ab = W.make_attention_batch(seed, B=5, Hq=Hq, Hkv=Hkv, d=16, prefix_range=prefix, n_range=(1, 12))
    np.testing.assert_allclose(OA.tree_attention(*_args(ab)), _sdpa(ab), atol=1e-12)


def test_chain_is_causal_attention():
    ab = W.make_attention_batch(4, B=3, Hq=2, Hkv=1, d=8, prefix_range=(0, 0),
                                parents=[W.chain_parents(n) for n in (1, 5, 9)])
    np.testing.assert_allclose(OA.tree_attention(*_args(ab)), _sdpa(ab, causal_chain=True), atol=1e-12)


def test_root_without_prefix_returns_its_value_and_equal_keys_average():
    ab = W.make_attention_batch(5, B=2, Hq=2, Hkv=1, d=8, prefix_range=(0, 0), parents=[[-1], [-1, 0, 0, 1]])
    o = OA.tree_attention(*_args(ab))
    np.testing.assert_array_equal(o[0, 0], _f64(ab.v)[0, 0])
    # identical keys: every visible key scores the same, so o = mean of the visible values
    args = list(_args(ab))
    args[1] = np.broadcast_to(args[1][:1], args[1].shape).copy()
    o = OA.tree_attention(*args)
    v = args[2]
    np.testing.assert_allclose(o[4, 1], (v[1, 0] + v[2, 0] + v[4, 0]) / 3, atol=1e-14)  # node 3: path 0, 1, 3
    args = list(_args(ab))
    args[8] = 0.0  # zero scale: uniform weights as well
    np.testing.assert_allclose(OA.tree_attention(*args)[3, 0], (v[1, 0] + v[3, 0]) / 2, atol=1e-14)


def test_branch_extraction_prefix_permutation_and_relabelling():
    rng = np.random.default_rng(0)
    ab = W.make_attention_batch(6, B=1, Hq=4, Hkv=2, d=8, prefix_range=(7, 7), n_range=(9, 9))
    o = OA.tree_attention(*_args(ab))
    q, k, v, kc, vc = (_f64(x) for x in (ab.q, ab.k, ab.v, ab.k_cache, ab.v_cache))
    for t in range(ab.T):
        path = []
        x = t
        while x >= 0:
            path.append(x)
            x = ab.parent[x]
        path = path[::-1]
        oc = OA.tree_attention(q[path], k[path], v[path], kc, vc, ab.cu_prefix, W.chain_parents(len(path)),
                               np.array([0, len(path)]), ab.scale)
        np.testing.assert_allclose(oc[-1], o[t], atol=1e-13)
    perm = rng.permutation(ab.P)
    o2 = OA.tree_attention(q, k, v, kc[perm], vc[perm], ab.cu_prefix, ab.parent, ab.cu_nodes, ab.scale)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    new_parent, order = W.random_topological_relabel(rng, ab.parent)
    o3 = OA.tree_attention(q[order], k[order], v[order], kc, vc, ab.cu_prefix, new_parent, ab.cu_nodes, ab.scale)
    np.testing.assert_allclose(o3, o[order], atol=1e-13)
