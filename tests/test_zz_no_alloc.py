"""gdn_tree_attention_noalloc: tree-bias attention for callers that cannot allocate device memory
(a serving engine whose allocator reserved the GPU's memory for its KV-cache pool at start-up, or
a framework that forbids allocation inside a forward step). Instead of a caller workspace it uses
a fixed scratch array built into the library, shared by every call.

The GPU test calls it twice in a row through the C ABI, on two different inputs whose key splits
use the scratch, and checks each output against gdn_tree_attention given its own workspace,
within the attention tolerance of the other tests (2^-8 max|v| from bf16 probabilities). It runs
alone in a fresh process as well as after the rest of the suite. The CPU test checks that sizes
needing more scratch than the built-in 32 MiB are refused before anything runs.
"""

import ctypes

import numpy as np
import pytest
import torch

from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import workloads as W

SCRATCH_BYTES = 32 << 20


def _bf(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _i32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def _both(ab):
    """The same inputs through gdn_tree_attention (own workspace) and gdn_tree_attention_noalloc."""
    ins = [_bf(ab.q), _bf(ab.k), _bf(ab.v), _bf(ab.k_cache), _bf(ab.v_cache), _i32(ab.cu_prefix), _i32(ab.parent),
           _i32(ab.cu_nodes)]
    sizes = (ab.B, ab.Hq, ab.Hkv, ab.T, ab.P, ab.d, ab.max_nodes, ab.max_prefix, ab.scale)
    need = gb.gdn_tree_attention_workspace_size(ab.B, ab.Hq, ab.Hkv, ab.d, ab.max_nodes, ab.max_prefix)
    assert 0 < need <= SCRATCH_BYTES  # the shape splits its keys, so the scratch is in use
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o_ref = torch.full((ab.T, ab.Hq, ab.d), float("nan"), device="cuda")
    o_new = torch.full((ab.T, ab.Hq, ab.d), float("nan"), device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    gb.gdn_tree_attention(*ins, *sizes, o_ref, ws, need, st)
    gb.gdn_tree_attention_noalloc(*ins, *sizes, o_new, st)
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0
    return o_ref.cpu().numpy(), o_new.cpu().numpy()


def _tol(ab):
    vmax = max(float(np.abs(W.bf16_bits_to_f32(ab.v)).max()), float(np.abs(W.bf16_bits_to_f32(ab.v_cache)).max()))
    return 2.0 ** -8 * vmax + 1e-5


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    first = W.make_attention_batch(71, B=2, Hq=16, Hkv=2, d=128, prefix_range=(2500, 3000), n_range=(4, 20))
    second = W.make_attention_batch(72, B=3, Hq=8, Hkv=2, d=64, prefix_range=(900, 1700), n_range=(1, 40))
    for ab in (first, second, first):  # the scratch keeps the previous call's contents
        o_ref, o_new = _both(ab)
        assert np.all(np.isfinite(o_new))
        assert float(np.max(np.abs(o_new - o_ref))) <= _tol(ab)


def test_sizes_beyond_the_scratch_are_refused():
    FAKE = 0x10000  # never dereferenced: the size check comes first
    B, Hq, Hkv, d, max_nodes, max_prefix = 64, 16, 2, 128, 32, 4096
    assert gb.gdn_tree_attention_workspace_size(B, Hq, Hkv, d, max_nodes, max_prefix) > SCRATCH_BYTES
    rc = gb.library().gdn_tree_attention_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, Hq, Hkv, 8, 64, d,
                                                 max_nodes, max_prefix, ctypes.c_float(0.1), FAKE, None, None)
    assert rc == gb.GDN_ETOOBIG
    rc = gb.library().gdn_tree_attention_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 12, 4, 8, 64, d,
                                                 max_nodes, max_prefix, ctypes.c_float(0.1), FAKE, None, None)
    assert rc == gb.GDN_EINVAL  # 3 query heads per key head
