"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 replay oracle.

Covers all five synthetic workload presets at their full sizes, compared with the oracle over the
whole output tensors (o, U, G) and the whole committed state (the tolerances are stated as a max
over a configuration's outputs and a Frobenius norm over its batch state), tiny and ragged random trees in
random topological orders, empty requests, the deepest (chain of 64) and widest (star of 64)
trees, forests, every verify kernel (gdn_tree_verify takes the register-resident streaming
kernel when max_nodes <= 8 and the tensor-core kernel above that; gdn_tree_verify_simt is the
CUDA-core kernel), the store-all comparison kernels, and the device-side error reporting.
"""

import numpy as np
import pytest
import torch

from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import device as gd
from gated_deltanet_tree_03_b300 import workloads as W
from gpu_util import check_commit, check_verify, run_gpu

pytestmark = pytest.mark.gpu

KERNELS = ["wy", "simt"]


@pytest.mark.parametrize("kernel", KERNELS + ["storeall"])
def test_chain3_d32_full(kernel):
    tb = W.make_config(0)
    res = run_gpu(tb, verify=kernel)
    assert res["status"] == 0
    check_verify(tb, res, tag=f"chain3_d32/{kernel}")
    check_commit(tb, res, tag=f"chain3_d32/{kernel}")


@pytest.mark.parametrize("kernel,max_nodes", [("wy", None), ("wy", 16), ("simt", None)])
def test_chain4_B256_full(kernel, max_nodes):
    """Depth-3 chain (4 nodes), B=256, H=32, d=128: the streaming kernel (max_nodes = 4) and the
    tensor-core kernel (16)."""
    tb = W.make_config(1)  # B=256, H=32, d=128, chain of 4
    res = run_gpu(tb, verify=kernel, max_nodes=max_nodes)
    assert res["status"] == 0
    check_verify(tb, res, tag=f"chain4_B256/{kernel}")
    check_commit(tb, res, tag=f"chain4_B256/{kernel}")


@pytest.mark.parametrize("batch", [1, 64])
@pytest.mark.parametrize("kernel,max_nodes", [("wy", None), ("wy", 32), ("simt", None)])
def test_rootbranch6_full(batch, kernel, max_nodes):
    tb = W.make_config(2, batch=batch)
    res = run_gpu(tb, verify=kernel, max_nodes=max_nodes)
    assert res["status"] == 0
    check_verify(tb, res, tag=f"rootbranch6/B{batch}/{kernel}")
    check_commit(tb, res, tag=f"rootbranch6/B{batch}/{kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_ragged16to64_B128_full(kernel):
    tb = W.make_config(3)
    res = run_gpu(tb, verify=kernel)
    assert res["status"] == 0
    check_verify(tb, res, tag=f"ragged16to64/{kernel}")
    check_commit(tb, res, tag=f"ragged16to64/{kernel}")


@pytest.mark.parametrize("batch", [1, 8, 32, 128, 256, 512])
def test_tree32_full(batch):
    """The batch sweep of 32-node trees, every batch size, one of its 48 layers' input sets each."""
    tb = W.make_config(4, batch=batch, layer=batch % 48)
    res = run_gpu(tb, verify="wy")
    assert res["status"] == 0
    check_verify(tb, res, tag=f"tree32/B{batch}")
    check_commit(tb, res, tag=f"tree32/B{batch}")


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("kernel", KERNELS + ["storeall"])
def test_random_ragged_trees(d, kernel):
    tb = W.make_random_batch(seed=100 + d, B=9, H=3, d=d, n_range=(1, 64), fanout_max=4, depth_max=8,
                             empty_every=4)
    res = run_gpu(tb, verify=kernel)
    assert res["status"] == 0
    check_verify(tb, res, tag=f"random/d{d}/{kernel}")
    check_commit(tb, res, tag=f"random/d{d}/{kernel}")


@pytest.mark.parametrize("shape", ["chain64", "star64", "forest"])
@pytest.mark.parametrize("kernel", KERNELS)
def test_extreme_shapes(shape, kernel):
    rng = np.random.default_rng(7)
    if shape == "chain64":
        parents = [W.chain_parents(64), W.chain_parents(33)]
        paths = [list(range(64)), list(range(20))]
    elif shape == "star64":
        parents = [np.array([-1] + [0] * 63, np.int32)]
        paths = [[0, 17]]
    else:  # several roots per request, random topological order
        p = np.array([-1, -1, 0, 1, 2, -1, 3, 5, 5, 6], np.int32)
        p, _ = W.random_topological_relabel(rng, p)
        parents = [p]
        leaf = W.leaves(p)[0]
        paths = [W.root_path(p, leaf)]
    tb = W.build_batch(rng, parents, paths, H=2, dk=128, dv=128)
    res = run_gpu(tb, verify=kernel)
    assert res["status"] == 0
    check_verify(tb, res, tag=f"{shape}/{kernel}")
    check_commit(tb, res, tag=f"{shape}/{kernel}")


def test_kernels_agree_and_snapshots_are_states():
    """Tensor-core WY, CUDA-core WY and store-all agree; store-all snapshots are replay states."""
    import oracle
    tb = W.make_random_batch(seed=5, B=4, H=2, d=64, n_range=(4, 20))
    a = run_gpu(tb, verify="wy", commit=False)
    b = run_gpu(tb, verify="simt", commit=False)
    c = run_gpu(tb, verify="storeall", commit=False)
    scale = np.max(np.abs(c["o"])) + 1
    assert np.max(np.abs(a["o"] - b["o"])) <= 2e-3 * scale
    assert np.max(np.abs(a["o"] - c["o"])) <= 2e-3 * scale
    inp = oracle.batch_inputs(tb)
    for r in range(tb.B):
        par = tb.request_parent(r)
        for t in range(len(par)):
            pth = W.root_path(par, t)
            path = np.full((tb.B, 64), -1, np.int32)
            plen = np.zeros(tb.B, np.int32)
            path[r, :len(pth)] = pth
            plen[r] = len(pth)
            ref = oracle.commit(inp["ST0"], inp["k"], inp["v"], inp["beta"], inp["g"], tb.parent, tb.cu_nodes,
                                path, plen, pairs=[r * tb.H + h for h in range(tb.H)])
            got = c["snap"][tb.cu_nodes[r] + t]
            rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
            assert rel <= 1e-4


@pytest.mark.parametrize("kernel", KERNELS + ["storeall"])
def test_bad_tree_reports_and_skips_only_that_request(kernel):
    tb = W.make_random_batch(seed=9, B=3, H=2, d=32, n_range=(5, 9))
    tb.parent[tb.cu_nodes[1] + 3] = 3  # node 3 of request 1 names itself as parent
    tb.path_len[:] = 0
    res = run_gpu(tb, verify=kernel, commit=False)
    assert res["status"] & gb.STATUS_BAD_TREE
    r1 = slice(tb.cu_nodes[1], tb.cu_nodes[2])
    assert np.all(np.isnan(res["o"][r1])) and np.all(np.isnan(res["U"][r1]))
    for r in (0, 2):
        rs = slice(tb.cu_nodes[r], tb.cu_nodes[r + 1])
        assert np.all(np.isfinite(res["o"][rs]))


@pytest.mark.parametrize("kernel", ["wy", "storeall"])
def test_bad_path_reports_and_keeps_state(kernel):
    tb = W.make_config(2, batch=4, heads=2)
    tb.path[1, :2] = [0, 4]  # 4 is a grandchild of 0, not a child
    tb.path_len[1] = 2
    tb.path[2, :1] = [3]  # does not start at the root
    tb.path_len[2] = 1
    res = run_gpu(tb, verify=kernel)
    assert res["status"] & gb.STATUS_BAD_PATH
    np.testing.assert_array_equal(res["ST"][1], tb.ST0[1])
    np.testing.assert_array_equal(res["ST"][2], tb.ST0[2])
    for r in (0, 3):
        if tb.path_len[r]:
            assert not np.array_equal(res["ST"][r], tb.ST0[r])


def test_too_many_nodes_and_empty_path():
    tb = W.make_random_batch(seed=10, B=3, H=2, d=64, n_range=(10, 12))
    tb.path_len[:] = 0
    res = run_gpu(tb, verify="wy", max_nodes=9)  # every request has more than 9 nodes
    assert res["status"] & gb.STATUS_TOO_MANY_NODES
    assert np.all(np.isnan(res["o"]))
    np.testing.assert_array_equal(res["ST"], tb.ST0)  # path_len == 0 keeps the state bit for bit


def test_host_argument_errors():
    tb = W.make_config(0)
    d = gd.upload(tb)
    out = gd.alloc_outputs(tb)
    base = [d["ST"], d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"], d["cu_nodes"], 1, 1, 3, 32, 32, 3,
            out["o"], out["U"], out["G"]]
    bad = list(base)
    bad[13] = 65
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_tree_verify(*bad)
    assert e.value.code == gb.GDN_ETOOBIG
    bad = list(base)
    bad[11] = 48
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_tree_verify(*bad)
    assert e.value.code == gb.GDN_EINVAL
    bad = list(base)
    bad[0] = d["ST"].data_ptr() + 4
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_tree_verify(*bad)
    assert e.value.code == gb.GDN_EALIGN
    # B == 0 launches nothing and succeeds
    empty = list(base)
    empty[8] = 0
    gb.gdn_tree_verify(*empty)
    torch.cuda.synchronize()


@pytest.mark.parametrize("dk,dv", [(128, 64), (64, 128), (32, 128), (128, 32)])
def test_mixed_key_value_widths(dk, dv):
    rng = np.random.default_rng(dk + dv)
    parents = [W.random_tree_parents(rng, int(n), 3, 6) for n in (5, 17, 40)]
    paths = [W.root_path(p, W.leaves(p)[-1]) for p in parents]
    tb = W.build_batch(rng, parents, paths, H=3, dk=dk, dv=dv)
    for kernel in KERNELS:
        res = run_gpu(tb, verify=kernel)
        assert res["status"] == 0
        check_verify(tb, res, tag=f"dk{dk}/dv{dv}/{kernel}")
        check_commit(tb, res, tag=f"dk{dk}/dv{dv}/{kernel}")


def test_oversized_max_nodes():
    """Node capacity far above the actual tree sizes (the node tile spans neighbouring requests)."""
    tb = W.make_config(2, batch=64, heads=4)
    padded = np.full((tb.B, 64), -1, np.int32)  # path rows are max_path apart
    padded[:, :tb.path.shape[1]] = tb.path
    tb.path = padded
    res = run_gpu(tb, verify="wy", max_nodes=64)
    assert res["status"] == 0
    check_verify(tb, res, tag="rootbranch6/max_nodes64")
    check_commit(tb, res, tag="rootbranch6/max_nodes64")


@pytest.mark.parametrize("kernel", KERNELS + ["storeall"])
def test_bad_offsets_reported(kernel):
    tb = W.make_random_batch(seed=11, B=3, H=2, d=64, n_range=(4, 6))
    T = tb.T
    tb.cu_nodes[2] = T + 5  # request 1 runs past the allocated rows, request 2 has negative size
    tb.path_len[:] = 0
    res = run_gpu(tb, verify=kernel, commit=False)
    assert res["status"] & gb.STATUS_BAD_OFFSETS
    r0 = slice(0, tb.cu_nodes[1])
    assert np.all(np.isfinite(res["o"][r0]))


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (64, 128), (128, 64), (32, 128), (32, 64)])
@pytest.mark.parametrize("nmax", [4, 6, 8])
def test_small_trees_streaming_kernel(dk, dv, nmax):
    """Trees of at most 8 nodes (forests, random topological orders, empty requests) take the
    register-resident streaming kernel; each of its node capacities (4, 6 and 8)."""
    rng = np.random.default_rng(1000 + dk + dv + nmax)
    parents, paths = [], []
    for r in range(13):
        if r % 5 == 4:
            parents.append(np.zeros(0, np.int32))
            paths.append([])
            continue
        n = int(rng.integers(1, nmax + 1))
        p = W.random_tree_parents(rng, n, fanout_max=3, depth_max=7)
        if r % 3 == 1 and n > 2:  # a forest: cut one edge
            p = p.copy()
            p[int(rng.integers(1, n))] = -1
        p, _ = W.random_topological_relabel(rng, p)
        parents.append(p)
        leaf = W.leaves(p)[int(rng.integers(len(W.leaves(p))))]
        full = W.root_path(p, leaf)
        paths.append(full[:int(rng.integers(0, len(full) + 1))])
    tb = W.build_batch(rng, parents, paths, H=3, dk=dk, dv=dv)
    res = run_gpu(tb, verify="wy", max_nodes=nmax)
    assert res["status"] == 0
    check_verify(tb, res, tag=f"stream/dk{dk}/dv{dv}/n{nmax}")
    check_commit(tb, res, tag=f"stream/dk{dk}/dv{dv}/n{nmax}")


def test_small_trees_streaming_kernel_errors():
    """Bad parent, too many nodes and bad offsets on the streaming path: reported, and only the
    affected request is skipped."""
    tb = W.make_random_batch(seed=12, B=4, H=2, d=128, n_range=(3, 6))
    tb.parent[tb.cu_nodes[1] + 2] = 2  # node 2 of request 1 names itself
    tb.path_len[:] = 0
    res = run_gpu(tb, verify="wy", commit=False, max_nodes=6)
    assert res["status"] & gb.STATUS_BAD_TREE
    r1 = slice(tb.cu_nodes[1], tb.cu_nodes[2])
    assert np.all(np.isnan(res["o"][r1]))
    for r in (0, 2, 3):
        rs = slice(tb.cu_nodes[r], tb.cu_nodes[r + 1])
        assert np.all(np.isfinite(res["o"][rs]))
    tb2 = W.make_random_batch(seed=13, B=3, H=2, d=128, n_range=(5, 7))
    tb2.path_len[:] = 0
    res = run_gpu(tb2, verify="wy", commit=False, max_nodes=4)
    assert res["status"] & gb.STATUS_TOO_MANY_NODES
    assert np.all(np.isnan(res["o"]))
