"""GPU: the serving-layout entry points (gdn_tree_verify_ex, gdn_tree_commit_ex,
gdn_tree_commit_verify_ex) against the fp64 serving-layout oracle - states in a slot pool with
padding requests, grouped q/k heads, a query scale and gates formed from their pre-activations -
through each verify kernel (streaming, tensor-core, CUDA-core at d = 32) and the fused
commit + verify kernel."""

import numpy as np
import pytest
import torch

from oracle import serving
from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import workloads as W
from gpu_util import G_TOL, O_TOL, S_TOL

pytestmark = pytest.mark.gpu


def _dev(x, dtype=None):
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def _upload(tb, sv, gates):
    d = {"pool": _dev(sv.pool), "slot": _dev(sv.slot.astype(np.int32)), "q": _dev(sv.q), "k": _dev(sv.k),
         "v": _dev(tb.v), "parent": _dev(tb.parent.astype(np.int32)), "cu": _dev(tb.cu_nodes.astype(np.int32)),
         "path": _dev(tb.path.astype(np.int32)), "plen": _dev(tb.path_len.astype(np.int32))}
    if gates:
        d.update(a_raw=_dev(sv.a_raw), b_raw=_dev(sv.b_raw), A_log=_dev(sv.A_log), dt_bias=_dev(sv.dt_bias))
        d["beta"] = d["g"] = None  # formed in the kernels
        lay = gb.layout(d["slot"], sv.pool.shape[0], sv.H_qk, sv.q_scale, d["a_raw"], d["b_raw"], d["A_log"],
                        d["dt_bias"])
    else:
        d["beta"], d["g"] = _dev(tb.beta), _dev(tb.g)
        lay = gb.layout(d["slot"], sv.pool.shape[0], sv.H_qk, sv.q_scale)
    return d, lay


def _outputs(tb):
    T = max(tb.T, 1)
    return {"o": torch.full((T, tb.H, tb.dv), float("nan"), device="cuda"),
            "U": torch.full((T, tb.H, tb.dv), float("nan"), device="cuda"),
            "G": torch.full((T, tb.H), float("nan"), device="cuda"),
            "status": torch.zeros(4, dtype=torch.int32, device="cuda")}


def _oracle_args(tb, sv):
    return (sv.pool, sv.slot, W.bf16_bits_to_f32(sv.q), W.bf16_bits_to_f32(sv.k), tb.v_f32(), tb.beta, tb.g,
            tb.parent, tb.cu_nodes)


def _check_outputs(tb, got, ref, tag, q_scale):
    """o within the output tolerance of the UNSCALED output (the scale is one final multiply, so
    the bound is taken on o / q_scale), U within the same bound, G within the gate-sum bound;
    rows of padding or rejected requests untouched (still NaN)."""
    o_ref, U_ref, G_ref = ref
    live = np.isfinite(G_ref[:, 0])
    for name, x, r, sc in (("o", got["o"], o_ref, q_scale), ("U", got["U"], U_ref, 1.0)):
        x = x[:tb.T]
        assert np.all(np.isnan(x[~live])), f"{tag}: {name} written for a padding or rejected request"
        assert np.all(np.isfinite(x[live])), f"{tag}: non-finite {name}"
        if live.any():
            e = float(np.max(np.abs(x[live].astype(np.float64) - r[live]))) / sc
            m = float(np.max(np.abs(r[live]))) / sc
            assert e <= O_TOL * (m + 1), f"{tag}: {name} max err {e:.3e} (max |ref| {m:.3f}, unscaled)"
    G = got["G"][:tb.T]
    assert np.all(np.isnan(G[~live]))
    assert np.all(np.abs(G[live].astype(np.float64) - G_ref[live]) <= G_TOL * (np.abs(G_ref[live]) + 1)), tag


def _check_pool(pool_before, pool_after, ref, touched, tag):
    for s in range(pool_before.shape[0]):
        if s in touched:
            rel = np.linalg.norm(pool_after[s] - ref[s]) / np.linalg.norm(ref[s])
            assert rel <= S_TOL, f"{tag}: slot {s} rel err {rel:.3e}"
        else:
            assert np.array_equal(pool_after[s], pool_before[s]), f"{tag}: slot {s} (not in the batch) changed"


CASES = [  # (tag, d, H, H_qk, n_range, gates, pad_every)
    ("streaming_d128_gqa4_gates", 128, 8, 2, (1, 8), True, 5),
    ("streaming_d64_plainheads", 64, 4, 4, (1, 6), False, 3),
    ("tensorcore_d128_gqa4_gates", 128, 4, 1, (9, 40), True, 4),
    ("tensorcore_d64_gqa2", 64, 4, 2, (9, 64), False, 0),
    ("cudacore_d32_gates", 32, 4, 2, (1, 20), True, 3),
]


@pytest.mark.parametrize("tag,d,H,H_qk,n_range,gates,pad_every", CASES, ids=[c[0] for c in CASES])
def test_verify_commit_ex_match_serving_oracle(tag, d, H, H_qk, n_range, gates, pad_every):
    tb, sv = W.make_serving_batch(seed=d + H + H_qk, B=11, H=H, H_qk=H_qk, d=d, n_range=n_range,
                                  pad_every=pad_every, empty_every=7)
    dv, lay = _upload(tb, sv, gates)
    out = _outputs(tb)
    gb.gdn_tree_verify_ex(dv["pool"], dv["q"], dv["k"], dv["v"], dv["beta"], dv["g"], dv["parent"], dv["cu"], tb.B,
                          tb.H, tb.T, d, d, tb.max_nodes, lay, out["o"], out["U"], out["G"], out["status"])
    torch.cuda.synchronize()
    got = {key: t.cpu().numpy() for key, t in out.items()}
    assert int(got["status"][0]) == 0
    ref = serving.verify(*_oracle_args(tb, sv), q_scale=sv.q_scale, gates=sv.gates if gates else None)
    _check_outputs(tb, got, ref, tag, sv.q_scale)
    gb.gdn_tree_commit_ex(dv["pool"], out["U"], out["G"], dv["k"], dv["parent"], dv["cu"], dv["path"], dv["plen"],
                          tb.B, tb.H, tb.T, d, d, tb.max_path, lay, out["status"])
    torch.cuda.synchronize()
    assert int(out["status"][0].item()) == 0
    pool_ref = serving.commit(sv.pool, sv.slot, W.bf16_bits_to_f32(sv.k), tb.v_f32(), tb.beta, tb.g, tb.parent,
                              tb.cu_nodes, tb.path, tb.path_len, gates=sv.gates if gates else None)
    touched = {int(s) for r, s in enumerate(sv.slot) if s >= 0 and tb.path_len[r] > 0}
    _check_pool(sv.pool, dv["pool"].cpu().numpy(), pool_ref, touched, tag)


@pytest.mark.parametrize("n_range", [(1, 8), (9, 30)], ids=["streaming", "tensorcore"])
def test_bad_slot_is_reported_and_skipped(n_range):
    tb, sv = W.make_serving_batch(seed=31, B=6, H=4, H_qk=2, d=128, n_range=n_range)
    sv.slot[2] = sv.pool.shape[0] + 5  # outside the pool
    sv.slot[4] = -3                    # negative but not the padding marker
    dv, lay = _upload(tb, sv, True)
    out = _outputs(tb)
    gb.gdn_tree_verify_ex(dv["pool"], dv["q"], dv["k"], dv["v"], None, None, dv["parent"], dv["cu"], tb.B, tb.H,
                          tb.T, 128, 128, tb.max_nodes, lay, out["o"], out["U"], out["G"], out["status"])
    torch.cuda.synchronize()
    got = {key: t.cpu().numpy() for key, t in out.items()}
    assert int(got["status"][0]) == gb.STATUS_BAD_SLOT
    sv_ok = W.ServingInputs(**{**sv.__dict__, "slot": np.where((sv.slot >= 0) & (sv.slot < sv.pool.shape[0]),
                                                                 sv.slot, -1).astype(np.int32)})
    ref = serving.verify(*_oracle_args(tb, sv_ok), q_scale=sv.q_scale, gates=sv.gates)
    _check_outputs(tb, got, ref, "bad slot", sv.q_scale)
    before = dv["pool"].cpu().numpy()
    st2 = torch.zeros(4, dtype=torch.int32, device="cuda")
    gb.gdn_tree_commit_ex(dv["pool"], out["U"], out["G"], dv["k"], dv["parent"], dv["cu"], dv["path"], dv["plen"],
                          tb.B, tb.H, tb.T, 128, 128, tb.max_path, lay, st2)
    torch.cuda.synchronize()
    assert int(st2[0].item()) == gb.STATUS_BAD_SLOT
    after = dv["pool"].cpu().numpy()
    pool_ref = serving.commit(sv.pool, sv_ok.slot, W.bf16_bits_to_f32(sv.k), tb.v_f32(), tb.beta, tb.g, tb.parent,
                              tb.cu_nodes, tb.path, tb.path_len, gates=sv.gates)
    touched = {int(s) for r, s in enumerate(sv_ok.slot) if s >= 0 and tb.path_len[r] > 0}
    _check_pool(before, after, pool_ref, touched, "bad slot commit")


@pytest.mark.parametrize("n_range,depth_max", [((1, 8), 3), ((9, 24), 6)], ids=["fused", "two_kernels"])
def test_commit_verify_ex_matches_two_step_oracle(n_range, depth_max):
    """Step 1 verifies tree 1 on the pool; step 2 commits tree 1's accepted paths and verifies tree 2 on the
    updated states in one call (fused when the shapes allow). Both requests sets share the slots."""
    tb1, sv1 = W.make_serving_batch(seed=40, B=9, H=4, H_qk=2, d=128, n_range=n_range, pad_every=4,
                                    depth_max=depth_max)
    tb2, sv2 = W.make_serving_batch(seed=41, B=9, H=4, H_qk=2, d=128, n_range=n_range, pad_every=4,
                                    depth_max=depth_max)
    sv2 = W.ServingInputs(**{**sv2.__dict__, "slot": sv1.slot, "pool": sv1.pool})
    d1, lay = _upload(tb1, sv1, True)
    d2, lay2 = _upload(tb2, sv2, True)  # same slots; this step's gate pre-activations
    out1, out2 = _outputs(tb1), _outputs(tb2)
    pool = d1["pool"]
    gb.gdn_tree_verify_ex(pool, d1["q"], d1["k"], d1["v"], None, None, d1["parent"], d1["cu"], tb1.B, tb1.H, tb1.T,
                          128, 128, tb1.max_nodes, lay, out1["o"], out1["U"], out1["G"], out1["status"])
    gb.gdn_tree_commit_verify_ex(pool, out1["U"], out1["G"], d1["k"], d1["parent"], d1["cu"], d1["path"], d1["plen"],
                                 tb1.T, tb1.max_path, d2["q"], d2["k"], d2["v"], None, None, d2["parent"], d2["cu"],
                                 tb2.B, tb2.H, tb2.T, 128, 128, tb2.max_nodes, lay2, out2["o"], out2["U"], out2["G"],
                                 out2["status"])
    torch.cuda.synchronize()
    assert int(out1["status"][0].item()) == 0 and int(out2["status"][0].item()) == 0
    pool_ref = serving.commit(sv1.pool, sv1.slot, W.bf16_bits_to_f32(sv1.k), tb1.v_f32(), tb1.beta, tb1.g,
                              tb1.parent, tb1.cu_nodes, tb1.path, tb1.path_len, gates=sv1.gates)
    touched = {int(s) for r, s in enumerate(sv1.slot) if s >= 0 and tb1.path_len[r] > 0}
    _check_pool(sv1.pool, pool.cpu().numpy(), pool_ref, touched, "commit_verify_ex state")
    sv2_ref = W.ServingInputs(**{**sv2.__dict__, "pool": pool_ref})
    ref = serving.verify(*_oracle_args(tb2, sv2_ref), q_scale=sv2.q_scale, gates=sv2.gates)
    _check_outputs(tb2, {key: t.cpu().numpy() for key, t in out2.items()}, ref, "commit_verify_ex outputs",
                   sv2.q_scale)
