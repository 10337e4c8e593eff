"""GPU: draft budgeting on the device (gdn_tree_budget_topb, gdn_tree_grow_best_first) against the
budget oracle. Every output is compared exactly: the chosen counts, candidates, parents and
packed batches, and the fp32 survival / branch values (both sides form them with the same fp32
products). The grown trees are then verified by gdn_tree_verify as a ragged batch."""

import numpy as np
import pytest
import torch

import oracle
from oracle import budget as OB
from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import workloads as W
from gpu_util import O_TOL

pytestmark = pytest.mark.gpu


def _topb_gpu(p, budget, packed=True):
    R, K = p.shape
    dp = torch.from_numpy(np.ascontiguousarray(p)).cuda()
    n_sel = torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda")
    surv = torch.full((max(R * K, 1),), float("nan"), device="cuda")
    cu = torch.full((R + 1,), -7, dtype=torch.int32, device="cuda")
    par = torch.full((R + min(budget, R * K) + 1,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    gb.gdn_tree_budget_topb(dp, R, K, budget, n_sel, surv, cu if packed else None, par if packed else None, st)
    torch.cuda.synchronize()
    return (n_sel.cpu().numpy()[:R], surv.cpu().numpy()[:R * K].reshape(R, K), cu.cpu().numpy(),
            par.cpu().numpy(), int(st[0].item()))


@pytest.mark.parametrize("R,K,budget", [(1, 1, 1), (7, 3, 5), (256, 7, 768), (256, 7, 0), (256, 7, 5000),
                                        (300, 5, 1499), (1024, 16, 4096), (2340, 7, 9000), (1, 63, 40)])
def test_topb_matches_oracle_exactly(R, K, budget):
    rng = np.random.default_rng(R * 100 + K)
    p = W.draw_acceptance(rng, R, K)
    n, s, cu, par, st = _topb_gpu(p, budget)
    n_ref, s_ref, cu_ref, par_ref = OB.topb(p, budget)
    assert st == 0
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(n, n_ref)
    np.testing.assert_array_equal(cu, cu_ref)
    np.testing.assert_array_equal(par[:len(par_ref)], par_ref)


def test_topb_ties_and_invalid_probabilities():
    R, K = 40, 6
    p = np.full((R, K), 0.5, np.float32)  # every request identical: pure tie-breaking
    p[3] = 1.0
    p[5, 2] = np.nan
    p[6, 0] = 1.5
    p[7, 1] = -0.0
    p[8, 4] = -0.25
    for budget in (0, 1, 17, 100, 240):
        n, s, cu, par, st = _topb_gpu(p, budget)
        n_ref, s_ref, cu_ref, par_ref = OB.topb(p, budget)
        assert st == gb.STATUS_BAD_PROB
        np.testing.assert_array_equal(s, s_ref)
        np.testing.assert_array_equal(n, n_ref)
        np.testing.assert_array_equal(cu, cu_ref)
    n, *_ = _topb_gpu(p, 100, packed=False)
    np.testing.assert_array_equal(n, OB.topb(p, 100)[0])


def _grow_gpu(p, fanout, depth, thr, max_nodes):
    R, C = p.shape
    dp = torch.from_numpy(np.ascontiguousarray(p)).cuda()
    mk = lambda fill, dt: torch.full((max(R * max_nodes, 1),), fill, dtype=dt, device="cuda")
    n = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    par_l, cand, val = mk(-7, torch.int32), mk(-7, torch.int32), mk(float("nan"), torch.float32)
    cu = torch.full((R + 1,), -7, dtype=torch.int32, device="cuda")
    par = mk(-7, torch.int32)
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    gb.gdn_tree_grow_best_first(dp, R, fanout, depth, thr, max_nodes, n, par_l, cand, val, cu, par, st)
    torch.cuda.synchronize()
    sh = (R, max_nodes)
    return {"n_nodes": n.cpu().numpy(), "parent_local": par_l.cpu().numpy()[:R * max_nodes].reshape(sh),
            "cand": cand.cpu().numpy()[:R * max_nodes].reshape(sh), "value": val.cpu().numpy()[:R * max_nodes].reshape(sh),
            "cu_nodes": cu.cpu().numpy(), "parent": par.cpu().numpy(), "status": int(st[0].item())}


GROW = [(2, 5, 0.02, 64), (3, 4, 0.05, 32), (4, 5, 0.01, 64), (1, 9, 0.3, 64), (3, 7, 0.02, 64),
        (8, 4, 0.003, 64), (2, 12, 0.001, 64), (3, 5, 0.0, 64), (3, 5, 2.0, 64), (3, 5, 0.02, 1), (3, 5, 0.02, 0)]


@pytest.mark.parametrize("fanout,depth,thr,max_nodes", GROW)
def test_grow_matches_oracle_exactly(fanout, depth, thr, max_nodes):
    rng = np.random.default_rng(fanout * 1000 + depth)
    R = 37
    p = W.draw_edge_probs(rng, R, fanout, depth)
    p[:, 1::7] = 0.25  # exactly repeated values: ties between siblings and cousins
    got = _grow_gpu(p, fanout, depth, thr, max_nodes)
    ref = OB.grow_best_first(p, fanout, depth, thr, max_nodes)
    assert got["status"] == 0
    for key in ("n_nodes", "cand", "parent_local", "value", "cu_nodes"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    np.testing.assert_array_equal(got["parent"][:len(ref["parent"])], ref["parent"])


def test_grow_invalid_probabilities_count_as_zero():
    rng = np.random.default_rng(5)
    p = W.draw_edge_probs(rng, 4, 3, 3)
    p[0, 1], p[1, 2], p[2, 5] = np.nan, 1.25, -0.5
    got = _grow_gpu(p, 3, 3, 0.0, 64)
    ref = OB.grow_best_first(p, 3, 3, 0.0, 64)
    assert got["status"] == gb.STATUS_BAD_PROB
    for key in ("n_nodes", "cand", "parent_local", "value"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)


def test_grown_trees_feed_verify():
    """Trees grown on the device are a valid ragged batch for gdn_tree_verify; its outputs match the
    oracle's replay of the same trees."""
    rng = np.random.default_rng(9)
    R, H, d = 24, 2, 64
    p = W.draw_edge_probs(rng, R, 3, 6)
    got = _grow_gpu(p, 3, 6, 0.01, 40)
    T = int(got["cu_nodes"][-1])
    parent, cu = got["parent"][:T].astype(np.int32), got["cu_nodes"].astype(np.int32)
    assert np.all(np.diff(cu) >= 1)
    tb = W.build_batch(rng, [parent[cu[r]:cu[r + 1]] for r in range(R)], [[0]] * R, H=H, dk=d, dv=d)
    from gated_deltanet_tree_03_b300 import device as gd
    din = gd.upload(tb)
    out = gd.alloc_outputs(tb, fill=float("nan"))
    gb.gdn_tree_verify(din["ST"], din["q"], din["k"], din["v"], din["beta"], din["g"], din["parent"],
                       din["cu_nodes"], R, H, T, d, d, tb.max_nodes, out["o"], out["U"], out["G"], out["status"])
    torch.cuda.synchronize()
    assert int(out["status"][0].item()) == 0
    o_ref, _, _ = oracle.verify(**oracle.batch_inputs(tb))
    o = out["o"][:T].cpu().numpy()
    assert np.max(np.abs(o - o_ref)) <= O_TOL * (np.max(np.abs(o_ref)) + 1)
