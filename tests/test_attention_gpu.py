"""GPU: tree-bias attention (gdn_tree_attention) against the fp64 oracle.

Tolerance: the kernel's scores and softmax are fp32, and its probabilities enter the P.V
product rounded to bf16 (relative error <= 2^-8 each). The output is a weighted mean of the
visible values, so |o - o_ref| <= 2^-8 max|v|; the test uses that bound (plus 1e-5 for the fp32
accumulation) over every output.
"""

import numpy as np
import pytest
import torch

from oracle import attention as OA
from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import workloads as W

pytestmark = pytest.mark.gpu


def _bf(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _run(ab, workspace=True, max_nodes=None, max_prefix=None, parent=None):
    mn = ab.max_nodes if max_nodes is None else max_nodes
    mp = ab.max_prefix if max_prefix is None else max_prefix
    o = torch.full((max(ab.T, 1), ab.Hq, ab.d), float("nan"), device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    i32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()
    ws, nb = None, 0
    if workspace:
        nb = gb.gdn_tree_attention_workspace_size(ab.B, ab.Hq, ab.Hkv, ab.d, mn, mp)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    kc = _bf(ab.k_cache) if ab.P else None
    vc = _bf(ab.v_cache) if ab.P else None
    gb.gdn_tree_attention(_bf(ab.q), _bf(ab.k), _bf(ab.v), kc, vc, i32(ab.cu_prefix),
                          i32(ab.parent if parent is None else parent), i32(ab.cu_nodes), ab.B, ab.Hq, ab.Hkv, ab.T,
                          ab.P, ab.d, mn, mp, ab.scale, o, ws, nb, st)
    torch.cuda.synchronize()
    return o[:ab.T].cpu().numpy(), int(st[0].item())


def _ref(ab):
    f = lambda x: W.bf16_bits_to_f32(x).astype(np.float64)
    return OA.tree_attention(f(ab.q), f(ab.k), f(ab.v), f(ab.k_cache), f(ab.v_cache), ab.cu_prefix, ab.parent,
                             ab.cu_nodes, ab.scale)


def _check(ab, o, tag):
    ref = _ref(ab)
    vmax = max(float(np.abs(W.bf16_bits_to_f32(ab.v)).max()),
               float(np.abs(W.bf16_bits_to_f32(ab.v_cache)).max()) if ab.P else 0.0)
    assert np.all(np.isfinite(o)), tag
    err = float(np.max(np.abs(o - ref)))
    assert err <= 2.0 ** -8 * vmax + 1e-5, f"{tag}: max err {err:.3e} (bound {2.0 ** -8 * vmax:.3e})"
    return err


CASES = [  # (tag, B, Hq, Hkv, d, prefix_range, n_range)
    ("d128_g8_short", 5, 16, 2, 128, (0, 300), (1, 12)),
    ("d128_g8_tiles", 3, 16, 2, 128, (100, 700), (30, 64)),   # up to 4 query tiles
    ("d128_g1", 4, 4, 4, 128, (1, 260), (1, 40)),
    ("d64_g4", 4, 8, 2, 64, (0, 513), (1, 33)),
    ("d128_g16_long", 2, 16, 1, 128, (2000, 5000), (2, 20)),  # many key blocks, split
    ("d128_no_prefix", 6, 8, 2, 128, (0, 0), (1, 64)),
]


@pytest.mark.parametrize("tag,B,Hq,Hkv,d,prefix,n_range", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("workspace", [True, False], ids=["split", "nosplit"])
def test_tree_attention_matches_oracle(tag, B, Hq, Hkv, d, prefix, n_range, workspace):
    ab = W.make_attention_batch(sum(map(ord, tag)), B=B, Hq=Hq, Hkv=Hkv, d=d, prefix_range=prefix, n_range=n_range,
                                fanout_max=3, depth_max=8)
    o, st = _run(ab, workspace=workspace)
    assert st == 0
    print(tag, "split" if workspace else "nosplit", "max err", _check(ab, o, tag))


def test_root_branch_tree_with_chain_and_relabelled_order():
    parents = [W.root_branch_parents(), W.chain_parents(9), W.random_topological_relabel(
        np.random.default_rng(1), W.random_tree_parents(np.random.default_rng(2), 40, 4, 8))[0]]
    ab = W.make_attention_batch(11, B=3, Hq=16, Hkv=2, d=128, prefix_range=(129, 640), parents=parents)
    o, st = _run(ab)
    assert st == 0
    _check(ab, o, "mixed trees")


def test_errors_are_reported_and_requests_skipped():
    ab = W.make_attention_batch(12, B=3, Hq=8, Hkv=2, d=128, prefix_range=(10, 200), n_range=(3, 10))
    bad = ab.parent.copy()
    bad[ab.cu_nodes[1] + 1] = 5  # request 1: node 1 names a later node as parent
    o, st = _run(ab, parent=bad)
    assert st == gb.STATUS_BAD_TREE
    ref = _ref(ab)
    for r in (0, 2):
        sl = slice(ab.cu_nodes[r], ab.cu_nodes[r + 1])
        assert np.max(np.abs(o[sl] - ref[sl])) <= 2.0 ** -8 * 5
    assert np.all(np.isnan(o[ab.cu_nodes[1]:ab.cu_nodes[2]]))
    o, st = _run(ab, max_prefix=int(np.diff(ab.cu_prefix).min()) - 1)  # a prefix longer than max_prefix
    assert st & gb.STATUS_BAD_OFFSETS


@pytest.mark.parametrize("Hq,Hkv,n_range", [(64, 2, (1, 16)), (128, 1, (1, 20))], ids=["g32", "g128"])
def test_wide_query_groups(Hq, Hkv, n_range):
    """Query-head groups of 32 and 128 (4 nodes, then 1 node, per 128-row tile: up to 20 tiles)."""
    ab = W.make_attention_batch(40 + Hq, B=3, Hq=Hq, Hkv=Hkv, d=128, prefix_range=(64, 400), n_range=n_range)
    for ws in (True, False):
        o, st = _run(ab, workspace=ws)
        assert st == 0
        _check(ab, o, f"G={Hq // Hkv} {'split' if ws else 'nosplit'}")


def test_bounds_larger_than_the_data():
    """max_nodes / max_prefix above the actual sizes: the extra tiles and key splits find no rows
    or no keys and must leave the result unchanged."""
    ab = W.make_attention_batch(51, B=4, Hq=16, Hkv=2, d=128, prefix_range=(0, 500), n_range=(1, 9))
    o_tight, st1 = _run(ab)
    o_loose, st2 = _run(ab, max_nodes=64, max_prefix=6000)
    assert st1 == 0 and st2 == 0
    _check(ab, o_loose, "loose bounds")
    assert float(np.max(np.abs(o_loose - o_tight))) <= 2.0 ** -8 * 5


def test_tiles_without_rows_leave_at_once():
    """Requests much smaller than the batch's largest leave query tiles without rows (here 16
    query heads per key/value head: 8 nodes fill a tile, so a 3-node request has two empty tiles
    out of three). Those CTAs return after their checks; none may wait out the kernel's 1 s
    bound on a copy it never issued. Also checks the results of such a batch."""
    import time
    ab = W.make_attention_batch(91, B=6, Hq=16, Hkv=1, d=128, prefix_range=(200, 900), n_range=(2, 24))
    assert ab.max_nodes > 16 and int(np.min(np.diff(ab.cu_nodes))) <= 8  # some tiles have no rows
    o, st = _run(ab)  # warm-up (module load, kernel attributes)
    assert st == 0
    t = time.perf_counter()
    o, st = _run(ab)
    dt = time.perf_counter() - t
    assert st == 0
    assert dt < 0.25, f"{dt:.3f} s for one small call"
    _check(ab, o, "row-less tiles")

