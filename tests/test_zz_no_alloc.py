"""gdn_tree_attention_noalloc: tree-bias attention for callers that cannot allocate device memory
(a serving engine whose allocator reserved the GPU's memory for its KV-cache pool at start-up, or
a framework that forbids allocation inside a forward step). Instead of a caller workspace it uses
a fixed scratch array built into the library, shared by every call.

The GPU tests call it through the C ABI:
  * twice in a row (and the first input again) on inputs whose key splits use the scratch. Each
    output must equal, bit for bit, gdn_tree_attention given a workspace of its own: same kernel,
    same split plan, so any partial write or stale read of the shared scratch shows. One call
    is also compared with the fp64 attention oracle (2^-8 max|v|, the bf16-probability bound);
  * on a shape whose full split plan needs more than the 32 MiB scratch: it runs with the plan
    that fits, equals bit for bit gdn_tree_attention given a 32 MiB workspace (the same plan),
    and agrees with the unsplit call within the bf16-probability bound;
  * once more in a fresh Python process, so that the scratch's first use on a device (the
    address lookup) is exercised in a process that has run nothing else.
The CPU test checks that invalid shapes are refused before anything runs.
"""

import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import workloads as W

SCRATCH_BYTES = 32 << 20
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bf(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _i32(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def _run(ab, workspace: str):
    """The same inputs through gdn_tree_attention (workspace "full": its own buffer of the planned
    size; "scratch": a buffer as large as the built-in scratch; "none": no workspace) and through
    gdn_tree_attention_noalloc."""
    import torch
    ins = [_bf(ab.q), _bf(ab.k), _bf(ab.v), _bf(ab.k_cache), _bf(ab.v_cache), _i32(ab.cu_prefix), _i32(ab.parent),
           _i32(ab.cu_nodes)]
    sizes = (ab.B, ab.Hq, ab.Hkv, ab.T, ab.P, ab.d, ab.max_nodes, ab.max_prefix, ab.scale)
    need = gb.gdn_tree_attention_workspace_size(ab.B, ab.Hq, ab.Hkv, ab.d, ab.max_nodes, ab.max_prefix)
    o_ref = torch.full((ab.T, ab.Hq, ab.d), float("nan"), device="cuda")
    o_new = torch.full((ab.T, ab.Hq, ab.d), float("nan"), device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    if workspace in ("full", "scratch"):
        nb = need if workspace == "full" else SCRATCH_BYTES
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        gb.gdn_tree_attention(*ins, *sizes, o_ref, ws, nb, st)
    else:
        gb.gdn_tree_attention(*ins, *sizes, o_ref, None, 0, st)
    gb.gdn_tree_attention_noalloc(*ins, *sizes, o_new, st)
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0
    return need, o_ref.cpu().numpy(), o_new.cpu().numpy()


def _tol(ab):
    vmax = max(float(np.abs(W.bf16_bits_to_f32(ab.v)).max()), float(np.abs(W.bf16_bits_to_f32(ab.v_cache)).max()))
    return 2.0 ** -8 * vmax + 1e-5


def _oracle(ab):
    from oracle import attention as OA
    f = lambda x: W.bf16_bits_to_f32(x).astype(np.float64)
    return OA.tree_attention(f(ab.q), f(ab.k), f(ab.v), f(ab.k_cache), f(ab.v_cache), ab.cu_prefix, ab.parent,
                             ab.cu_nodes, ab.scale)


def two_calls_in_a_row() -> None:
    """Body of the two-call check (also run by the fresh-process test)."""
    first = W.make_attention_batch(71, B=2, Hq=16, Hkv=2, d=128, prefix_range=(2500, 3000), n_range=(4, 20))
    second = W.make_attention_batch(72, B=3, Hq=8, Hkv=2, d=64, prefix_range=(900, 1700), n_range=(1, 40))
    for i, ab in enumerate((first, second, first)):  # the scratch keeps the previous call's contents
        need, o_ref, o_new = _run(ab, "full")
        assert 0 < need <= SCRATCH_BYTES  # the shape splits its keys, so the scratch is in use
        assert np.all(np.isfinite(o_new))
        np.testing.assert_array_equal(o_new, o_ref)
        if i == 1:
            assert float(np.max(np.abs(o_new - _oracle(ab)))) <= _tol(ab)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    two_calls_in_a_row()


@pytest.mark.gpu
def test_noalloc_plans_within_the_scratch():
    """7 requests x 16384-key prefixes, 32 query / 4 key-value heads, 64-node trees: 112 (request,
    head, tile) CTAs, whose best split plan needs about 37 MB. The scratch takes the best plan that
    fits in 32 MiB."""
    rng = np.random.default_rng(73)
    parents = [W.random_tree_parents(rng, 64, 3, 6) for _ in range(7)]
    ab = W.make_attention_batch(73, B=7, Hq=32, Hkv=4, d=128, prefix_range=(16384, 16384), parents=parents)
    need, o_ref, o_new = _run(ab, "scratch")
    assert need > SCRATCH_BYTES
    assert np.all(np.isfinite(o_new))
    np.testing.assert_array_equal(o_new, o_ref)
    _, o_unsplit, _ = _run(ab, "none")
    assert float(np.max(np.abs(o_new - o_unsplit))) <= _tol(ab)


@pytest.mark.gpu
def test_noalloc_in_a_fresh_process():
    code = ("import sys; sys.path.insert(0, 'tests'); sys.path.insert(0, '.'); "
            "import test_zz_no_alloc as t; t.two_calls_in_a_row(); print('fresh ok')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "fresh ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_invalid_shapes_are_refused():
    FAKE = 0x10000  # never dereferenced: the shape checks come first
    lib = gb.library()
    d, max_nodes, max_prefix = 128, 32, 4096
    rc = lib.gdn_tree_attention_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 12, 4, 8, 64, d,
                                        max_nodes, max_prefix, ctypes.c_float(0.1), FAKE, None, None)
    assert rc == gb.GDN_EINVAL  # 3 query heads per key head
    rc = lib.gdn_tree_attention_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 16, 2, 8, 64, d,
                                        65, max_prefix, ctypes.c_float(0.1), FAKE, None, None)
    assert rc == gb.GDN_ETOOBIG  # more than 64 nodes per request
    rc = lib.gdn_tree_attention_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 16, 2, 8, 64, d,
                                        max_nodes, max_prefix, ctypes.c_float(-1.0), FAKE, None, None)
    assert rc == gb.GDN_EINVAL  # the score scale must be positive
