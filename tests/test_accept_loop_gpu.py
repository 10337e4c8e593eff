"""GPU: device-side greedy acceptance (bit-exact against the oracle) and the closed
verify -> accept -> commit loop over many rounds, with the fp32 device state checked against the
fp64 oracle state carried through the same accepted paths."""

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import device as gd
from gated_deltanet_tree_03_b300 import workloads as W
from gpu_util import O_TOL, S_TOL

pytestmark = pytest.mark.gpu


def _accept_gpu(draft, target, parent, cu, B, T, max_nodes, max_path):
    dev = "cuda"
    d_draft = torch.from_numpy(np.ascontiguousarray(draft, np.int32)).to(dev)
    d_target = torch.from_numpy(np.ascontiguousarray(target, np.int32)).to(dev)
    d_parent = torch.from_numpy(np.ascontiguousarray(parent, np.int32)).to(dev)
    d_cu = torch.from_numpy(np.ascontiguousarray(cu, np.int32)).to(dev)
    path = torch.full((max(B, 1), max(max_path, 1)), -7, dtype=torch.int32, device=dev)
    plen = torch.full((max(B, 1),), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    gb.gdn_tree_accept_greedy(d_draft if T else None, d_target if T else None, d_parent if T else None, d_cu, B, T,
                              max_nodes, max_path, path, plen, status)
    torch.cuda.synchronize()
    return path.cpu().numpy()[:B, :max_path], plen.cpu().numpy()[:B], int(status[0].item())


@pytest.mark.parametrize("seed,n_range,vocab", [(1, (1, 8), 4), (2, (1, 64), 6), (3, (30, 64), 3), (4, (1, 20), 50)])
def test_accept_matches_oracle_exactly(seed, n_range, vocab):
    rng = np.random.default_rng(seed)
    tb = W.make_random_batch(seed=seed, B=37, H=1, d=8, n_range=n_range, fanout_max=4, depth_max=8, empty_every=6)
    draft, target = W.draw_tokens(rng, tb.parent, tb.cu_nodes, vocab=vocab, p_match=0.8)
    path, plen, status = _accept_gpu(draft, target, tb.parent, tb.cu_nodes, tb.B, tb.T, max(tb.max_nodes, 1), 64)
    ref_path, ref_len, ref_trunc = oracle.accept_greedy(draft, target, tb.parent, tb.cu_nodes, 64)
    assert status == 0
    np.testing.assert_array_equal(plen, ref_len)
    np.testing.assert_array_equal(path, ref_path)


def test_accept_truncation_bad_tree_and_offsets():
    parents = [W.chain_parents(6), np.array([-1, 0, 0], np.int32), W.chain_parents(4)]
    cu = np.array([0, 6, 9, 13], np.int32)
    parent = np.concatenate(parents)
    draft = np.arange(13, dtype=np.int32)
    target = np.roll(draft, -1)  # every chain node's target is its child's draft
    path, plen, status = _accept_gpu(draft, target, parent, cu, 3, 13, 6, 3)
    ref_path, ref_len, ref_trunc = oracle.accept_greedy(draft, target, parent, cu, 3)
    np.testing.assert_array_equal(plen, ref_len)
    np.testing.assert_array_equal(path, ref_path)
    assert ref_trunc[0] and status & gb.STATUS_PATH_TRUNCATED
    bad = parent.copy()
    bad[6 + 2] = 2  # node 2 of request 1 names itself
    path, plen, status = _accept_gpu(draft, target, bad, cu, 3, 13, 6, 8)
    assert status & gb.STATUS_BAD_TREE and plen[1] == 0 and np.all(path[1] == -1)
    assert plen[0] == 6 and plen[2] == 4
    off = cu.copy()
    off[2] = 20  # request 1 runs past T
    path, plen, status = _accept_gpu(draft, target, parent, off, 3, 13, 64, 8)
    assert status & gb.STATUS_BAD_OFFSETS and plen[1] == 0


@pytest.mark.parametrize("rounds,n_range,tag", [(100, (2, 8), "streaming"), (40, (9, 24), "tensor-core")])
def test_verify_accept_commit_loop_tracks_fp64_replay(rounds, n_range, tag):
    """Closed decode loop on the device: every round a fresh draft tree is verified against the
    current state, the accepted path is found on the device and committed in place. The oracle
    replays the same rounds in fp64 from its own state; paths must agree exactly and the fp32
    state must stay within the committed-state tolerance of the fp64 one throughout."""
    B, H, d = 6, 2, 64
    rng = np.random.default_rng(77)
    state = None
    state_ref = None
    worst = 0.0
    for rnd in range(rounds):
        tb = W.make_random_batch(seed=9000 + rnd, B=B, H=H, d=d, n_range=n_range, fanout_max=3, depth_max=6,
                                 shuffle_order=False)
        if state is None:
            state = torch.from_numpy(tb.ST0.copy()).cuda()
            state_ref = tb.ST0.astype(np.float64)
        draft, target = W.draw_tokens(rng, tb.parent, tb.cu_nodes, vocab=5, p_match=0.75)
        din = gd.upload(tb)
        out = gd.alloc_outputs(tb, fill=float("nan"))
        mp = tb.max_nodes
        gb.gdn_tree_verify(state, din["q"], din["k"], din["v"], din["beta"], din["g"], din["parent"], din["cu_nodes"],
                           B, H, tb.T, d, d, mp, out["o"], out["U"], out["G"], out["status"])
        d_draft = torch.from_numpy(draft).cuda()
        d_target = torch.from_numpy(target).cuda()
        path = torch.empty((B, mp), dtype=torch.int32, device="cuda")
        plen = torch.empty((B,), dtype=torch.int32, device="cuda")
        gb.gdn_tree_accept_greedy(d_draft, d_target, din["parent"], din["cu_nodes"], B, tb.T, mp, mp, path, plen,
                                  out["status"])
        o_dev = out["o"][:tb.T].clone()
        gb.gdn_tree_commit(state, out["U"], out["G"], din["k"], din["parent"], din["cu_nodes"], path, plen, B, H,
                           tb.T, d, d, mp, out["status"])
        torch.cuda.synchronize()
        assert int(out["status"][0].item()) == 0
        ref_path, ref_len, _ = oracle.accept_greedy(draft, target, tb.parent, tb.cu_nodes, mp)
        np.testing.assert_array_equal(plen.cpu().numpy(), ref_len)
        np.testing.assert_array_equal(path.cpu().numpy(), ref_path)
        inp = oracle.batch_inputs(tb)
        if rnd % 10 == 0:
            o_ref, _, _ = oracle.verify(state_ref, inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], tb.parent,
                                        tb.cu_nodes)
            err = float(np.max(np.abs(o_dev.cpu().numpy() - o_ref)))
            assert err <= O_TOL * (float(np.max(np.abs(o_ref))) + 1), f"{tag} round {rnd}: output error {err}"
        state_ref = oracle.commit(state_ref, inp["k"], inp["v"], inp["beta"], inp["g"], tb.parent, tb.cu_nodes,
                                  ref_path, ref_len)
        rel = float(np.linalg.norm(state.cpu().numpy() - state_ref) / np.linalg.norm(state_ref))
        worst = max(worst, rel)
        assert rel <= S_TOL, f"{tag} round {rnd}: state drift {rel:.3e}"
    print(f"{tag}: worst relative state drift over {rounds} rounds {worst:.2e}")
