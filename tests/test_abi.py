"""C ABI checks that need no GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching CUDA."""

import ctypes

import pytest

from gated_deltanet_tree_03_b300 import binding as gb

EXPECTED = {"gdn_tree_verify", "gdn_tree_verify_simt", "gdn_tree_commit", "gdn_tree_verify_storeall",
            "gdn_tree_commit_storeall", "gdn_tree_accept_greedy", "gdn_tree_commit_verify", "gdn_status_str",
            "gdn_abi_version", "gdn_tree_verify_ex", "gdn_tree_commit_ex", "gdn_tree_commit_verify_ex",
            "gdn_tree_budget_topb", "gdn_tree_grow_best_first", "gdn_tree_attention",
            "gdn_tree_attention_workspace_size", "gdn_tree_attention_noalloc"}


def test_header_declares_expected_symbols():
    assert EXPECTED <= set(gb.declared_symbols())


def test_every_declared_symbol_is_exported():
    lib = gb.library()
    for name in gb.declared_symbols():
        assert hasattr(lib, name), f"{name} declared in include/gdn_tree.h but not exported"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version():
    assert gb.abi_version() == 3
    for code in (gb.GDN_OK, gb.GDN_EINVAL, gb.GDN_ETOOBIG, gb.GDN_EALIGN, gb.GDN_ECUDA, gb.GDN_EARCH):
        assert gb.status_str(code).startswith("GDN_")
    assert "unknown" in gb.status_str(99)


FAKE = 0x10000  # 16-byte aligned host-side stand-in address; never dereferenced (checks fail first)


def _verify(fn, **kw):
    args = dict(ST=FAKE, q=FAKE, k=FAKE, v=FAKE, beta=FAKE, g=FAKE, parent=FAKE, cu_nodes=FAKE, B=1, H=1,
                T=4, d_k=32, d_v=32, max_nodes=4, o=FAKE, U=FAKE, G=FAKE, status=None)
    args.update(kw)
    return fn(args["ST"], args["q"], args["k"], args["v"], args["beta"], args["g"], args["parent"],
              args["cu_nodes"], args["B"], args["H"], args["T"], args["d_k"], args["d_v"], args["max_nodes"],
              args["o"], args["U"], args["G"], args["status"], None)


@pytest.mark.parametrize("name", ["gdn_tree_verify", "gdn_tree_verify_simt"])
@pytest.mark.parametrize("kw,code", [
    (dict(d_k=48), gb.GDN_EINVAL), (dict(d_v=256), gb.GDN_EINVAL), (dict(H=0), gb.GDN_EINVAL),
    (dict(B=-1), gb.GDN_EINVAL), (dict(max_nodes=65), gb.GDN_ETOOBIG), (dict(q=None), gb.GDN_EINVAL),
    (dict(o=FAKE + 4), gb.GDN_EALIGN), (dict(status=FAKE + 8), gb.GDN_EALIGN), (dict(B=0), gb.GDN_OK),
    (dict(B=70000), gb.GDN_EINVAL), (dict(T=-1), gb.GDN_EINVAL), (dict(T=0, q=None), gb.GDN_OK)])
def test_verify_host_checks(name, kw, code):
    fn = getattr(gb.library(), name)
    assert _verify(fn, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(max_path=65), gb.GDN_ETOOBIG), (dict(d_k=16), gb.GDN_EINVAL), (dict(path=None), gb.GDN_EINVAL),
    (dict(U=FAKE + 2), gb.GDN_EALIGN), (dict(B=0), gb.GDN_OK)])
def test_commit_host_checks(kw, code):
    args = dict(ST=FAKE, U=FAKE, G=FAKE, k=FAKE, parent=FAKE, cu_nodes=FAKE, path=FAKE, path_len=FAKE, B=1,
                H=1, T=4, d_k=32, d_v=32, max_path=4, status=None)
    args.update(kw)
    rc = gb.library().gdn_tree_commit(*[args[x] for x in ("ST", "U", "G", "k", "parent", "cu_nodes", "path",
                                                          "path_len", "B", "H", "T", "d_k", "d_v", "max_path",
                                                          "status")], None)
    assert rc == code


def test_binding_raises_on_error():
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_tree_verify(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 48, 32, 4, FAKE, FAKE, FAKE,
                           stream=0)
    assert e.value.code == gb.GDN_EINVAL


@pytest.mark.parametrize("kw,code", [
    (dict(max_path=65), gb.GDN_ETOOBIG), (dict(max_nodes=65), gb.GDN_ETOOBIG), (dict(B=-1), gb.GDN_EINVAL),
    (dict(path=None), gb.GDN_EINVAL), (dict(draft=None), gb.GDN_EINVAL), (dict(path_len=FAKE + 4), gb.GDN_EALIGN),
    (dict(B=0), gb.GDN_OK)])
def test_accept_host_checks(kw, code):
    args = dict(draft=FAKE, target=FAKE, parent=FAKE, cu_nodes=FAKE, B=1, T=4, max_nodes=4, max_path=4, path=FAKE,
                path_len=FAKE, status=None)
    args.update(kw)
    rc = gb.library().gdn_tree_accept_greedy(*[args[x] for x in ("draft", "target", "parent", "cu_nodes", "B", "T",
                                                                 "max_nodes", "max_path", "path", "path_len",
                                                                 "status")], None)
    assert rc == code


def _layout(**kw):
    f = dict(state_slot=None, n_slots=0, H_qk=0, q_scale=1.0, a_raw=None, b_raw=None, A_log=None, dt_bias=None)
    f.update(kw)
    return gb.GdnLayout(f["state_slot"], f["n_slots"], f["H_qk"], f["q_scale"], f["a_raw"], f["b_raw"], f["A_log"],
                        f["dt_bias"])


GATES = dict(a_raw=FAKE, b_raw=FAKE, A_log=FAKE, dt_bias=FAKE)


@pytest.mark.parametrize("lay,kw,code", [
    (dict(H_qk=3), {}, gb.GDN_EINVAL),                       # 4 value heads are not a multiple of 3
    (dict(H_qk=-1), {}, gb.GDN_EINVAL),
    (dict(state_slot=FAKE, n_slots=0), {}, gb.GDN_EINVAL),  # a pool needs its size
    (dict(state_slot=FAKE + 4, n_slots=8), {}, gb.GDN_EALIGN),
    (dict(q_scale=float("inf")), {}, gb.GDN_EINVAL),
    (dict(q_scale=float("nan")), {}, gb.GDN_EINVAL),
    (dict(a_raw=FAKE), {}, gb.GDN_EINVAL),                   # some but not all gate arrays
    (dict(GATES, dt_bias=FAKE + 8), {}, gb.GDN_EALIGN),
    (dict(GATES), dict(beta=None, g=None, B=0), gb.GDN_OK),   # fused gates: beta and g are not read
    ({}, dict(beta=None), gb.GDN_EINVAL),                    # ... but are required otherwise
    (dict(H_qk=2, state_slot=FAKE, n_slots=3, q_scale=0.0), dict(B=0), gb.GDN_OK),
])
def test_verify_ex_layout_host_checks(lay, kw, code):
    args = dict(ST=FAKE, q=FAKE, k=FAKE, v=FAKE, beta=FAKE, g=FAKE, parent=FAKE, cu_nodes=FAKE, B=1, H=4, T=4,
                d_k=32, d_v=32, max_nodes=4, o=FAKE, U=FAKE, G=FAKE, status=None)
    args.update(kw)
    L = _layout(**lay)
    order = ("ST", "q", "k", "v", "beta", "g", "parent", "cu_nodes", "B", "H", "T", "d_k", "d_v", "max_nodes")
    rc = gb.library().gdn_tree_verify_ex(*[args[x] for x in order], ctypes.byref(L), args["o"], args["U"],
                                         args["G"], args["status"], None)
    assert rc == code


@pytest.mark.parametrize("lay,code", [
    (dict(H_qk=3), gb.GDN_EINVAL), (dict(state_slot=FAKE, n_slots=-2), gb.GDN_EINVAL),
    (dict(q_scale=float("inf"), a_raw=FAKE), gb.GDN_OK),  # commit ignores the scale and the gates
])
def test_commit_ex_layout_host_checks(lay, code):
    L = _layout(**lay)
    rc = gb.library().gdn_tree_commit_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 4, 32, 32, 4,
                                         ctypes.byref(L), None, None)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), gb.GDN_EINVAL), (dict(K=64), gb.GDN_EINVAL), (dict(budget=-1), gb.GDN_EINVAL),
    (dict(R=2341, K=7), gb.GDN_ETOOBIG), (dict(p=None), gb.GDN_EINVAL), (dict(n_sel=FAKE + 4), gb.GDN_EALIGN),
    (dict(R=16384, K=1), gb.GDN_ETOOBIG),  # 16384 items, but 256 KiB of shared memory for one CTA
    (dict(cu=None), gb.GDN_EINVAL),  # parent without cu_nodes
    (dict(R=0), gb.GDN_OK)])
def test_budget_topb_host_checks(kw, code):
    a = dict(p=FAKE, R=4, K=7, budget=5, n_sel=FAKE, surv=None, cu=FAKE, par=FAKE)
    a.update(kw)
    rc = gb.library().gdn_tree_budget_topb(a["p"], a["R"], a["K"], a["budget"], a["n_sel"], a["surv"], a["cu"],
                                           a["par"], None, None)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(fanout=0), gb.GDN_EINVAL), (dict(depth=-1), gb.GDN_EINVAL), (dict(max_nodes=65), gb.GDN_ETOOBIG),
    (dict(fanout=2, depth=13), gb.GDN_ETOOBIG), (dict(fanout=4, depth=7), gb.GDN_ETOOBIG),
    (dict(thr=float("nan")), gb.GDN_EINVAL), (dict(parent=None), gb.GDN_EINVAL),  # cu_nodes without parent
    (dict(parent_local=None), gb.GDN_EINVAL), (dict(R=0), gb.GDN_OK)])
def test_grow_host_checks(kw, code):
    a = dict(p=FAKE, R=4, fanout=3, depth=4, thr=0.1, max_nodes=32, n=FAKE, parent_local=FAKE, cu=FAKE, parent=FAKE)
    a.update(kw)
    rc = gb.library().gdn_tree_grow_best_first(a["p"], a["R"], a["fanout"], a["depth"], a["thr"], a["max_nodes"],
                                               a["n"], a["parent_local"], None, None, a["cu"], a["parent"], None, None)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(Hq=12, Hkv=4), gb.GDN_EINVAL),  # group of 3 query heads: not a power of two
    (dict(Hq=6, Hkv=4), gb.GDN_EINVAL), (dict(d=32), gb.GDN_EINVAL), (dict(max_nodes=65), gb.GDN_ETOOBIG),
    (dict(scale=float("inf")), gb.GDN_EINVAL), (dict(scale=0.0), gb.GDN_EINVAL), (dict(scale=-0.5), gb.GDN_EINVAL),
    (dict(q=None), gb.GDN_EINVAL), (dict(kc=None), gb.GDN_EINVAL),
    (dict(o=FAKE + 4), gb.GDN_EALIGN), (dict(B=0), gb.GDN_OK), (dict(max_nodes=0), gb.GDN_OK),
    (dict(kc=None, vc=None, P=0), gb.GDN_ECUDA)])  # valid arguments: only the missing GPU stops it
def test_attention_host_checks(kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, cp=FAKE, par=FAKE, cu=FAKE, B=2, Hq=16, Hkv=2, T=8, P=64, d=128,
             max_nodes=4, max_prefix=32, scale=0.1, o=FAKE)
    a.update(kw)
    rc = gb.library().gdn_tree_attention(a["q"], a["k"], a["v"], a["kc"], a["vc"], a["cp"], a["par"], a["cu"], a["B"],
                                         a["Hq"], a["Hkv"], a["T"], a["P"], a["d"], a["max_nodes"], a["max_prefix"],
                                         ctypes.c_float(a["scale"]), a["o"], None, 0, None, None)
    if code == gb.GDN_ECUDA:
        assert rc in (gb.GDN_ECUDA, gb.GDN_EARCH)
    else:
        assert rc == code


def test_attention_workspace_size_is_zero_without_splits():
    assert gb.gdn_tree_attention_workspace_size(0, 16, 2, 128, 8, 4096) == 0
    assert gb.gdn_tree_attention_workspace_size(4, 16, 2, 128, 8, 100) == 0  # one key block: nothing to split
    big = gb.gdn_tree_attention_workspace_size(1, 16, 2, 128, 6, 8192)
    assert big > 0 and big % (128 * 130 * 4) == 0


def test_attention_key_splits_follow_the_wave_model():
    """One CTA per SM: a grid that already fills whole waves stays unsplit, a small one splits.
    The bench's 4096-key batches (64 requests, 2 key/value heads) have 128 CTAs (6-node trees, one
    query tile) and 256 (32-node trees, two tiles); splitting either measured slower on B300."""
    assert gb.gdn_tree_attention_workspace_size(64, 16, 2, 128, 6, 4096) == 0
    assert gb.gdn_tree_attention_workspace_size(64, 16, 2, 128, 32, 4096) == 0
    per_tile = 128 * 130 * 4  # one partial tile: 128 rows of (d + 2) floats
    small = gb.gdn_tree_attention_workspace_size(1, 16, 2, 128, 6, 4096)  # 2 CTAs unsplit
    assert small > 0 and small % per_tile == 0 and small // per_tile > 2
    assert small // per_tile <= 148  # the split grid stays within one wave (here 2 x 32 = 64 CTAs)


def test_attention_workspace_stays_under_its_bound():
    """The key splits never plan more than 4 CTAs per SM, so the workspace stays under 4 x SMs x
    128 rows x (d + 2) floats: with the host's SM count unknown here, the planner assumes 148 SMs."""
    bound = lambda d: 4 * 148 * 128 * (d + 2) * 4
    for B in (1, 2, 5, 17, 64, 150, 300):
        for Hq, Hkv in ((16, 2), (8, 8), (32, 4), (4, 1)):
            for d in (64, 128):
                for mn in (1, 6, 32, 64):
                    for mp in (0, 100, 4096, 40000):
                        ws = gb.gdn_tree_attention_workspace_size(B, Hq, Hkv, d, mn, mp)
                        assert ws <= bound(d), (B, Hq, Hkv, d, mn, mp, ws)
                        assert ws % (128 * (d + 2) * 4) == 0
