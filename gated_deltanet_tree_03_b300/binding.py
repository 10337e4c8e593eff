"""Thin ctypes binding of libgdn_tree.so (declared in include/gdn_tree.h).

Argument marshalling only: every step of the computation runs in the CUDA kernels behind
the C ABI. Array arguments may be CUDA ``torch.Tensor`` objects (their device pointer is
passed), plain integer device addresses, or ``None`` (NULL). ``stream`` defaults to torch's
current CUDA stream. A non-GDN_OK return code raises ``GdnError``. If the shared library is
missing and cannot be built, importing this module raises - there is no fallback.
"""

from __future__ import annotations

import ctypes
import re
import os

from . import _build

GDN_OK, GDN_EINVAL, GDN_ETOOBIG, GDN_EALIGN, GDN_ECUDA, GDN_EARCH = 0, 1, 2, 3, 6, 7
STATUS_BAD_TREE, STATUS_BAD_PATH, STATUS_TOO_MANY_NODES, STATUS_TIMEOUT, STATUS_BAD_OFFSETS = 1, 2, 4, 8, 16
STATUS_PATH_TRUNCATED, STATUS_BAD_SLOT, STATUS_BAD_PROB, STATUS_OUT_OF_BOUNDS = 32, 64, 128, 256
MAX_NODES = 64

HEADER = os.path.join(_build.INCLUDE, "gdn_tree.h")


class GdnError(RuntimeError):
    def __init__(self, code: int, fn: str):
        self.code = int(code)
        super().__init__(f"{fn}: {status_str(code)}")


def _load() -> ctypes.CDLL:
    # GDN_TREE_DEBUG_BOUNDS=1 selects the address-checking build of the same kernels
    path = _build.build(debug_bounds=os.environ.get("GDN_TREE_DEBUG_BOUNDS") == "1")
    return ctypes.CDLL(path)


_lib = _load()

_P = ctypes.c_void_p
_I = ctypes.c_int32


class GdnLayout(ctypes.Structure):
    """``gdn_layout`` of gdn_tree.h (serving layout of the *_ex entry points)."""

    _fields_ = [("state_slot", _P), ("n_slots", _I), ("H_qk", _I), ("q_scale", ctypes.c_float),
                ("a_raw", _P), ("b_raw", _P), ("A_log", _P), ("dt_bias", _P)]


_LP = ctypes.POINTER(GdnLayout)

_SIGS = {
    "gdn_tree_verify": [_P] * 8 + [_I] * 6 + [_P] * 4 + [_P],
    "gdn_tree_verify_simt": [_P] * 8 + [_I] * 6 + [_P] * 4 + [_P],
    "gdn_tree_commit": [_P] * 8 + [_I] * 6 + [_P, _P],
    "gdn_tree_verify_storeall": [_P] * 8 + [_I] * 6 + [_P] * 5 + [_P],
    "gdn_tree_commit_storeall": [_P] * 6 + [_I] * 6 + [_P, _P],
    "gdn_tree_accept_greedy": [_P] * 4 + [_I] * 4 + [_P] * 3 + [_P],
    "gdn_tree_commit_verify": [_P] * 8 + [_I] * 2 + [_P] * 7 + [_I] * 6 + [_P] * 4 + [_P],
    "gdn_tree_verify_ex": [_P] * 8 + [_I] * 6 + [_LP] + [_P] * 4 + [_P],
    "gdn_tree_commit_ex": [_P] * 8 + [_I] * 6 + [_LP] + [_P, _P],
    "gdn_tree_commit_verify_ex": [_P] * 8 + [_I] * 2 + [_P] * 7 + [_I] * 6 + [_LP] + [_P] * 4 + [_P],
    "gdn_tree_budget_topb": [_P] + [_I] * 3 + [_P] * 5 + [_P],
    "gdn_tree_grow_best_first": [_P] + [_I] * 3 + [ctypes.c_float, _I] + [_P] * 7 + [_P],
    "gdn_tree_attention": [_P] * 8 + [_I] * 8 + [ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P],
    "gdn_tree_attention_noalloc": [_P] * 8 + [_I] * 8 + [ctypes.c_float, _P, _P, _P],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.gdn_tree_attention_workspace_size.argtypes = [_I] * 6
_lib.gdn_tree_attention_workspace_size.restype = ctypes.c_size_t
_lib.gdn_status_str.argtypes = [ctypes.c_int]
_lib.gdn_status_str.restype = ctypes.c_char_p
_lib.gdn_abi_version.argtypes = []
_lib.gdn_abi_version.restype = ctypes.c_int32


def declared_symbols() -> list[str]:
    """Names of every function the public header declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def library() -> ctypes.CDLL:
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("array arguments must be CUDA tensors (device memory)")
        if not x.is_contiguous():
            raise ValueError("array arguments must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a device pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_str(code: int) -> str:
    return _lib.gdn_status_str(int(code)).decode()


def abi_version() -> int:
    return int(_lib.gdn_abi_version())


def _check(rc: int, fn: str) -> None:
    if rc != GDN_OK:
        raise GdnError(rc, fn)


def gdn_tree_verify(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, o, U, G,
                    status=None, stream=None):
    _check(_lib.gdn_tree_verify(_ptr(ST), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(parent),
                                _ptr(cu_nodes), B, H, T, d_k, d_v, max_nodes, _ptr(o), _ptr(U), _ptr(G),
                                _ptr(status), _stream(stream)), "gdn_tree_verify")


def gdn_tree_verify_simt(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, o, U, G,
                         status=None, stream=None):
    _check(_lib.gdn_tree_verify_simt(_ptr(ST), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                     _ptr(parent), _ptr(cu_nodes), B, H, T, d_k, d_v, max_nodes, _ptr(o),
                                     _ptr(U), _ptr(G), _ptr(status), _stream(stream)),
           "gdn_tree_verify_simt")


def gdn_tree_commit(ST, U, G, k, parent, cu_nodes, path, path_len, B, H, T, d_k, d_v, max_path,
                    status=None, stream=None):
    _check(_lib.gdn_tree_commit(_ptr(ST), _ptr(U), _ptr(G), _ptr(k), _ptr(parent), _ptr(cu_nodes),
                                _ptr(path), _ptr(path_len), B, H, T, d_k, d_v, max_path, _ptr(status),
                                _stream(stream)), "gdn_tree_commit")


def gdn_tree_verify_storeall(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes,
                             snapshots, o, U, G, status=None, stream=None):
    _check(_lib.gdn_tree_verify_storeall(_ptr(ST), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                         _ptr(parent), _ptr(cu_nodes), B, H, T, d_k, d_v, max_nodes,
                                         _ptr(snapshots), _ptr(o), _ptr(U), _ptr(G), _ptr(status),
                                         _stream(stream)), "gdn_tree_verify_storeall")


def gdn_tree_commit_storeall(ST, snapshots, parent, cu_nodes, path, path_len, B, H, T, d_k, d_v, max_path,
                             status=None, stream=None):
    _check(_lib.gdn_tree_commit_storeall(_ptr(ST), _ptr(snapshots), _ptr(parent), _ptr(cu_nodes),
                                         _ptr(path), _ptr(path_len), B, H, T, d_k, d_v, max_path,
                                         _ptr(status), _stream(stream)), "gdn_tree_commit_storeall")


def gdn_tree_accept_greedy(draft_tok, target_tok, parent, cu_nodes, B, T, max_nodes, max_path, path, path_len,
                           status=None, stream=None):
    _check(_lib.gdn_tree_accept_greedy(_ptr(draft_tok), _ptr(target_tok), _ptr(parent), _ptr(cu_nodes), B, T,
                                       max_nodes, max_path, _ptr(path), _ptr(path_len), _ptr(status),
                                       _stream(stream)), "gdn_tree_accept_greedy")


def gdn_tree_commit_verify(ST, U_prev, G_prev, k_prev, parent_prev, cu_nodes_prev, path, path_len, T_prev, max_path,
                           q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, o, U, G, status=None,
                           stream=None):
    _check(_lib.gdn_tree_commit_verify(_ptr(ST), _ptr(U_prev), _ptr(G_prev), _ptr(k_prev), _ptr(parent_prev),
                                       _ptr(cu_nodes_prev), _ptr(path), _ptr(path_len), T_prev, max_path, _ptr(q),
                                       _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(parent), _ptr(cu_nodes), B, H, T,
                                       d_k, d_v, max_nodes, _ptr(o), _ptr(U), _ptr(G), _ptr(status),
                                       _stream(stream)), "gdn_tree_commit_verify")


def layout(state_slot=None, n_slots=0, H_qk=0, q_scale=1.0, a_raw=None, b_raw=None, A_log=None, dt_bias=None):
    """A ``GdnLayout`` from device arrays (torch CUDA tensors or addresses) and scalars."""
    return GdnLayout(_ptr(state_slot), int(n_slots), int(H_qk), float(q_scale), _ptr(a_raw), _ptr(b_raw),
                     _ptr(A_log), _ptr(dt_bias))


def _lay(lay):
    return None if lay is None else ctypes.byref(lay)


def gdn_tree_verify_ex(ST, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, lay, o, U, G,
                       status=None, stream=None):
    _check(_lib.gdn_tree_verify_ex(_ptr(ST), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(parent),
                                   _ptr(cu_nodes), B, H, T, d_k, d_v, max_nodes, _lay(lay), _ptr(o), _ptr(U),
                                   _ptr(G), _ptr(status), _stream(stream)), "gdn_tree_verify_ex")


def gdn_tree_commit_ex(ST, U, G, k, parent, cu_nodes, path, path_len, B, H, T, d_k, d_v, max_path, lay,
                       status=None, stream=None):
    _check(_lib.gdn_tree_commit_ex(_ptr(ST), _ptr(U), _ptr(G), _ptr(k), _ptr(parent), _ptr(cu_nodes), _ptr(path),
                                   _ptr(path_len), B, H, T, d_k, d_v, max_path, _lay(lay), _ptr(status),
                                   _stream(stream)), "gdn_tree_commit_ex")


def gdn_tree_commit_verify_ex(ST, U_prev, G_prev, k_prev, parent_prev, cu_nodes_prev, path, path_len, T_prev,
                              max_path, q, k, v, beta, g, parent, cu_nodes, B, H, T, d_k, d_v, max_nodes, lay, o, U,
                              G, status=None, stream=None):
    _check(_lib.gdn_tree_commit_verify_ex(_ptr(ST), _ptr(U_prev), _ptr(G_prev), _ptr(k_prev), _ptr(parent_prev),
                                          _ptr(cu_nodes_prev), _ptr(path), _ptr(path_len), T_prev, max_path, _ptr(q),
                                          _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(parent), _ptr(cu_nodes), B, H,
                                          T, d_k, d_v, max_nodes, _lay(lay), _ptr(o), _ptr(U), _ptr(G), _ptr(status),
                                          _stream(stream)), "gdn_tree_commit_verify_ex")


def gdn_tree_budget_topb(p_accept, R, K, budget, n_sel, survival=None, cu_nodes=None, parent=None, status=None,
                         stream=None):
    _check(_lib.gdn_tree_budget_topb(_ptr(p_accept), R, K, budget, _ptr(n_sel), _ptr(survival), _ptr(cu_nodes),
                                     _ptr(parent), _ptr(status), _stream(stream)), "gdn_tree_budget_topb")


def gdn_tree_grow_best_first(p_edge, R, fanout, depth, threshold, max_nodes, n_nodes, parent_local, cand=None,
                             value=None, cu_nodes=None, parent=None, status=None, stream=None):
    _check(_lib.gdn_tree_grow_best_first(_ptr(p_edge), R, fanout, depth, float(threshold), max_nodes, _ptr(n_nodes),
                                         _ptr(parent_local), _ptr(cand), _ptr(value), _ptr(cu_nodes), _ptr(parent),
                                         _ptr(status), _stream(stream)), "gdn_tree_grow_best_first")


def gdn_tree_attention_workspace_size(B, H_q, H_kv, d, max_nodes, max_prefix) -> int:
    return int(_lib.gdn_tree_attention_workspace_size(B, H_q, H_kv, d, max_nodes, max_prefix))


def gdn_tree_attention(q, k, v, k_cache, v_cache, cu_prefix, parent, cu_nodes, B, H_q, H_kv, T, P_total, d, max_nodes,
                       max_prefix, scale, o, workspace=None, workspace_bytes=0, status=None, stream=None):
    if workspace is not None and hasattr(workspace, "numel") and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.gdn_tree_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(cu_prefix),
                                   _ptr(parent), _ptr(cu_nodes), B, H_q, H_kv, T, P_total, d, max_nodes, max_prefix,
                                   float(scale), _ptr(o), _ptr(workspace), int(workspace_bytes), _ptr(status),
                                   _stream(stream)), "gdn_tree_attention")


def gdn_tree_attention_noalloc(q, k, v, k_cache, v_cache, cu_prefix, parent, cu_nodes, B, H_q, H_kv, T, P_total, d,
                               max_nodes, max_prefix, scale, o, status=None, stream=None):
    _check(_lib.gdn_tree_attention_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(cu_prefix),
                                           _ptr(parent), _ptr(cu_nodes), B, H_q, H_kv, T, P_total, d, max_nodes,
                                           max_prefix, float(scale), _ptr(o), _ptr(status), _stream(stream)),
           "gdn_tree_attention_noalloc")
