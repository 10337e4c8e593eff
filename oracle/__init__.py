"""CPU oracle for GDN draft-tree verify / commit (fp64 replay of the gated delta rule).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline / reference leg may import this package. The library path never does, and it
shares no code with the CUDA kernels.

Two implementations of the same definition:
  * ``gdn_oracle.c`` - plain C, fp64, OpenMP over (request, head) pairs; exposed here as
    ``verify`` / ``commit`` (optionally on a sampled list of pairs).
  * ``replay.py``    - a NumPy twin for small cases.

Greedy acceptance (``accept_greedy``) is plain Python loops over the tree.

Parity pins live in ``tests/test_oracle_pins.py`` and ``tests/test_accept_pins.py``: a hand-worked d=2 example
(``tests/golden/``), closed forms of the rule (no-write, pure decay, delta-rule erasure,
orthonormal keys), linearity, chain = sequential decode, branch extraction, topological
relabelling, and brute-force store-all stepping on tiny inputs.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import replay  # noqa: F401  (NumPy twin)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_OK, ORACLE_BAD_TREE, ORACLE_BAD_PATH, ORACLE_BAD_ARG = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc -O2 -fopenmp) if missing or older than its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            i = ctypes.c_int
            lib.gdn_oracle_verify.argtypes = [i, i, i, i, dp, dp, dp, dp, dp, dp, ip, ip, ip, i, dp, dp, dp, i]
            lib.gdn_oracle_verify.restype = i
            lib.gdn_oracle_commit.argtypes = [i, i, i, i, dp, dp, dp, dp, dp, ip, ip, ip, ip, i, ip, i, dp, i]
            lib.gdn_oracle_commit.restype = i
            lib.gdn_oracle_max_threads.argtypes = []
            lib.gdn_oracle_max_threads.restype = i
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _d(x):
    a = np.ascontiguousarray(x, dtype=np.float64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i(x):
    a = np.ascontiguousarray(x, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


class OracleError(ValueError):
    pass


def _pairs(pairs, B, H):
    if pairs is None:
        return None, None, B * H
    p, pp = _i(np.asarray(pairs, dtype=np.int32).reshape(-1))
    return p, pp, int(p.size)


def verify(ST0, q, k, v, beta, g, parent, cu_nodes, pairs=None, n_threads: int = 0):
    """Replay oracle for verify.

    ``pairs``: optional flat (r*H + h) indices; outputs are then compact - for each listed
    pair, in order, n_nodes(r) rows. Without ``pairs`` outputs are full [T,H,dv] / [T,H].
    """
    lib = _load()
    ST0a, ST0p = _d(ST0)
    B, H, dk, dv = ST0a.shape
    qa, qp = _d(q)
    ka, kp = _d(k)
    va, vp = _d(v)
    ba, bp = _d(beta)
    ga, gp = _d(g)
    pa, pp = _i(parent)
    ca, cp = _i(cu_nodes)
    pl, plp, npairs = _pairs(pairs, B, H)
    if pl is None:
        rows = int(ca[-1]) * H
    else:
        rows = int(sum(int(ca[x // H + 1] - ca[x // H]) for x in pl))
    o = np.zeros((rows, dv))
    U = np.zeros((rows, dv))
    G = np.zeros(rows)
    if pl is None:
        # full layout: compute pair by pair in (r, h) order, then scatter to [T, H, *]
        order = np.arange(B * H, dtype=np.int32)
        pl, plp = _i(order)
        npairs = B * H
    rc = lib.gdn_oracle_verify(B, H, dk, dv, ST0p, qp, kp, vp, bp, gp, pp, cp, plp, npairs,
                               o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                               U.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                               G.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(n_threads))
    if rc != ORACLE_OK:
        raise OracleError({1: "bad tree", 2: "bad path", 3: "bad argument"}.get(rc, str(rc)))
    if pairs is not None:
        return o, U, G
    T = int(ca[-1])
    of = np.zeros((T, H, dv))
    Uf = np.zeros((T, H, dv))
    Gf = np.zeros((T, H))
    row = 0
    for r in range(B):
        t0, t1 = int(ca[r]), int(ca[r + 1])
        for h in range(H):
            n = t1 - t0
            of[t0:t1, h] = o[row:row + n]
            Uf[t0:t1, h] = U[row:row + n]
            Gf[t0:t1, h] = G[row:row + n]
            row += n
    return of, Uf, Gf


def commit(ST0, k, v, beta, g, parent, cu_nodes, path, path_len, pairs=None, n_threads: int = 0):
    """Replay oracle for commit: the state after each request's accepted path.

    Returns [B,H,dk,dv] without ``pairs``; with ``pairs`` a compact [n_pairs, dk, dv].
    """
    lib = _load()
    ST0a, ST0p = _d(ST0)
    B, H, dk, dv = ST0a.shape
    ka, kp = _d(k)
    va, vp = _d(v)
    ba, bp = _d(beta)
    ga, gp = _d(g)
    pa, pp = _i(parent)
    ca, cp = _i(cu_nodes)
    path_a = np.ascontiguousarray(path, dtype=np.int32)
    if path_a.ndim == 1:
        path_a = path_a.reshape(B, -1)
    max_path = int(path_a.shape[1]) if path_a.size else 0
    if max_path == 0:
        path_a = np.full((B, 1), -1, dtype=np.int32)
        max_path = 1
    patha, pathp = _i(path_a)
    la, lp = _i(path_len)
    pl, plp, npairs = _pairs(pairs, B, H)
    out = np.zeros((npairs, dk, dv))
    rc = lib.gdn_oracle_commit(B, H, dk, dv, ST0p, kp, vp, bp, gp, pp, cp, pathp, lp, max_path, plp,
                               npairs, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(n_threads))
    if rc != ORACLE_OK:
        raise OracleError({1: "bad tree", 2: "bad path", 3: "bad argument"}.get(rc, str(rc)))
    if pairs is None:
        return out.reshape(B, H, dk, dv)
    return out


def accept_greedy(draft_tok, target_tok, parent, cu_nodes, max_path):
    """Greedy acceptance oracle (plain loops); see ``replay.accept_greedy``."""
    return replay.accept_greedy(draft_tok, target_tok, parent, cu_nodes, max_path)


def batch_inputs(tb):
    """fp64 views of a ``workloads.TreeBatch`` in the oracle's argument order (verify)."""
    return dict(ST0=tb.ST0.astype(np.float64), q=tb.q_f32().astype(np.float64),
                k=tb.k_f32().astype(np.float64), v=tb.v_f32().astype(np.float64),
                beta=tb.beta.astype(np.float64), g=tb.g.astype(np.float64),
                parent=tb.parent, cu_nodes=tb.cu_nodes)
