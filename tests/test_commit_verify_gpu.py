"""GPU: gdn_tree_commit_verify (the previous step's commit folded into this step's verify) against
gdn_tree_commit followed by gdn_tree_verify, and against the fp64 oracle doing the same two steps."""

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import device as gd
from gated_deltanet_tree_03_b300 import workloads as W
from gpu_util import O_TOL, S_TOL

pytestmark = pytest.mark.gpu


def _two_steps(tb1, tb2, fused, max_nodes2=None):
    """Step 1: verify tb1 on its state. Step 2: commit tb1's paths, verify tb2 (fused or not)."""
    d1, d2 = gd.upload(tb1), gd.upload(tb2)
    out1 = gd.alloc_outputs(tb1, fill=float("nan"))
    out2 = gd.alloc_outputs(tb2, fill=float("nan"))
    ST = d1["ST"]
    mn1, mn2 = tb1.max_nodes, tb2.max_nodes if max_nodes2 is None else max_nodes2
    gb.gdn_tree_verify(ST, d1["q"], d1["k"], d1["v"], d1["beta"], d1["g"], d1["parent"], d1["cu_nodes"], tb1.B, tb1.H,
                       tb1.T, tb1.dk, tb1.dv, mn1, out1["o"], out1["U"], out1["G"], out1["status"])
    args_prev = (out1["U"], out1["G"], d1["k"], d1["parent"], d1["cu_nodes"], d1["path"], d1["path_len"])
    args_new = (d2["q"], d2["k"], d2["v"], d2["beta"], d2["g"], d2["parent"], d2["cu_nodes"])
    if fused:
        gb.gdn_tree_commit_verify(ST, *args_prev, tb1.T, tb1.max_path, *args_new, tb2.B, tb2.H, tb2.T, tb2.dk, tb2.dv,
                                  mn2, out2["o"], out2["U"], out2["G"], out2["status"])
    else:
        gb.gdn_tree_commit(ST, *args_prev, tb1.B, tb1.H, tb1.T, tb1.dk, tb1.dv, tb1.max_path, out2["status"])
        gb.gdn_tree_verify(ST, *args_new, tb2.B, tb2.H, tb2.T, tb2.dk, tb2.dv, mn2, out2["o"], out2["U"], out2["G"],
                           out2["status"])
    torch.cuda.synchronize()
    return {"ST": ST.cpu().numpy(), "o": out2["o"][:tb2.T].cpu().numpy(), "U": out2["U"][:tb2.T].cpu().numpy(),
            "G": out2["G"][:tb2.T].cpu().numpy(), "status": int(out2["status"][0].item())}


def _pair(seed, B, H, d, n_range, paths_max=4, empty_every=0):
    tb1 = W.make_random_batch(seed=seed, B=B, H=H, d=d, n_range=n_range, fanout_max=3, depth_max=5,
                              shuffle_order=False)
    tb2 = W.make_random_batch(seed=seed + 1, B=B, H=H, d=d, n_range=n_range, fanout_max=3, depth_max=5,
                              empty_every=empty_every)
    tb2.ST0 = tb1.ST0
    # accepted paths of step 1: random root prefixes of at most paths_max nodes (some empty)
    rng = np.random.default_rng(seed)
    path = np.full((B, paths_max), -1, np.int32)
    plen = np.zeros(B, np.int32)
    for r in range(B):
        par = tb1.request_parent(r)
        full = W.root_path(par, W.leaves(par)[int(rng.integers(len(W.leaves(par))))])[:paths_max]
        L = int(rng.integers(0, len(full) + 1))
        path[r, :L] = full[:L]
        plen[r] = L
    tb1.path, tb1.path_len = path, plen
    return tb1, tb2


def _oracle_two_steps(tb1, tb2):
    i1, i2 = oracle.batch_inputs(tb1), oracle.batch_inputs(tb2)
    S1 = oracle.commit(i1["ST0"], i1["k"], i1["v"], i1["beta"], i1["g"], tb1.parent, tb1.cu_nodes, tb1.path,
                       tb1.path_len)
    o2, U2, _ = oracle.verify(S1, i2["q"], i2["k"], i2["v"], i2["beta"], i2["g"], tb2.parent, tb2.cu_nodes)
    return S1, o2, U2


@pytest.mark.parametrize("d,n_range,empty_every", [(128, (2, 4), 0), (128, (1, 6), 3), (64, (2, 8), 0),
                                                   (128, (6, 20), 0)])
def test_fused_equals_commit_then_verify_and_oracle(d, n_range, empty_every):
    tb1, tb2 = _pair(31 + d + n_range[1], B=11, H=3, d=d, n_range=n_range, empty_every=empty_every)
    fused = _two_steps(tb1, tb2, fused=True)
    sep = _two_steps(tb1, tb2, fused=False)
    assert fused["status"] == 0 and sep["status"] == 0
    S1, o2, U2 = _oracle_two_steps(tb1, tb2)
    for res, tag in ((fused, "fused"), (sep, "separate")):
        rel = np.linalg.norm(res["ST"] - S1) / np.linalg.norm(S1)
        assert rel <= S_TOL, f"{tag}: state {rel:.2e}"
        for name, x, ref in (("o", res["o"], o2), ("U", res["U"], U2)):
            err = float(np.max(np.abs(x - ref))) if ref.size else 0.0
            assert err <= O_TOL * (float(np.max(np.abs(ref))) + 1 if ref.size else 1), f"{tag} {name} {err:.2e}"
    np.testing.assert_allclose(fused["ST"], sep["ST"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(fused["o"], sep["o"], rtol=1e-4, atol=1e-5)


def test_fused_bad_path_keeps_state_and_bad_new_tree_still_commits():
    tb1, tb2 = _pair(5, B=4, H=2, d=128, n_range=(3, 4))
    tb1.path[1, :2] = [0, 0]  # node 0 is not its own child: not a root-to-node chain
    tb1.path_len[1] = 2
    tb2.parent[tb2.cu_nodes[2] + 1] = 1  # node 1 of request 2 names itself: bad new tree
    res = _two_steps(tb1, tb2, fused=True)
    assert res["status"] & gb.STATUS_BAD_PATH and res["status"] & gb.STATUS_BAD_TREE
    i1 = oracle.batch_inputs(tb1)
    ok_len = tb1.path_len.copy()
    ok_len[1] = 0
    S1 = oracle.commit(i1["ST0"], i1["k"], i1["v"], i1["beta"], i1["g"], tb1.parent, tb1.cu_nodes, tb1.path, ok_len)
    np.testing.assert_array_equal(res["ST"][1], tb1.ST0[1])  # rejected path: state untouched
    rel = np.linalg.norm(res["ST"][2] - S1[2]) / np.linalg.norm(S1[2])
    assert rel <= S_TOL  # request 2's new tree is malformed, its previous path is still committed
    r2 = slice(tb2.cu_nodes[2], tb2.cu_nodes[3])
    assert np.all(np.isnan(res["o"][r2]))


def test_fused_rejects_aliased_pseudo_values():
    tb1, tb2 = _pair(6, B=2, H=1, d=64, n_range=(2, 3))
    d1, d2 = gd.upload(tb1), gd.upload(tb2)
    out = gd.alloc_outputs(tb2)
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_tree_commit_verify(d1["ST"], out["U"], out["G"], d1["k"], d1["parent"], d1["cu_nodes"], d1["path"],
                                  d1["path_len"], tb1.T, tb1.max_path, d2["q"], d2["k"], d2["v"], d2["beta"], d2["g"],
                                  d2["parent"], d2["cu_nodes"], 2, 1, tb2.T, 64, 64, tb2.max_nodes, out["o"], out["U"],
                                  out["G"])
    assert e.value.code == gb.GDN_EINVAL
