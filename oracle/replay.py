"""NumPy twin of the fp64 replay oracle (small cases only).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's
CPU-baseline leg, never by the library path. It shares no code with the CUDA path.

It computes the plain definition:

    gated delta rule  S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t

replayed from the committed state along each node's root-to-node path (GDN Tree-Scan
abstract: a candidate row carries the state native sequential decode would produce along its
root-to-node path; TreeWY page, method section: a branch refers only to its ancestors).
The pseudo-value of node t is the one the TreeWY page's method section describes - the new
value minus what the preceding state predicts, scaled by beta:
u_t = b_t (v_t - a_t S_parent k_t). Commit replays the accepted path (TreeWY page, method
section: only the accepted path's state is rebuilt).

Inputs use the library layouts with fp64 values: ST0 [B,H,dk,dv], q,k [T,H,dk], v [T,H,dv],
beta,g [T,H], parent [T], cu_nodes [B+1], path [B,max_path], path_len [B].
"""

from __future__ import annotations

import numpy as np


def rule_step(S: np.ndarray, a: float, b: float, k: np.ndarray, v: np.ndarray):
    """One application of the rule to S (d_v x d_k). Returns (new S, pseudo-value u)."""
    Sk = S @ k
    u = b * (v - a * Sk)
    S_new = a * S - a * b * np.outer(Sk, k) + b * np.outer(v, k)
    return S_new, u


def _root_path(parent_r: np.ndarray, t: int) -> list[int]:
    path = []
    x = t
    while x >= 0:
        path.append(x)
        x = int(parent_r[x])
    return path[::-1]


def _check_tree(parent, cu_nodes):
    for r in range(len(cu_nodes) - 1):
        n = cu_nodes[r + 1] - cu_nodes[r]
        for t in range(n):
            p = parent[cu_nodes[r] + t]
            if p < -1 or p >= t:
                raise ValueError(f"request {r}: node {t} has parent {p}, not in [-1, {t - 1}]")


def _check_path(parent, cu_nodes, path, path_len):
    for r in range(len(cu_nodes) - 1):
        n = cu_nodes[r + 1] - cu_nodes[r]
        L = int(path_len[r])
        if L < 0 or L > n or L > path.shape[1]:
            raise ValueError(f"request {r}: path length {L} out of range")
        prev = -1
        for i in range(L):
            x = int(path[r, i])
            if x < 0 or x >= n or parent[cu_nodes[r] + x] != prev:
                raise ValueError(f"request {r}: accepted path is not a root-to-node chain")
            prev = x


def verify(ST0, q, k, v, beta, g, parent, cu_nodes):
    """Per-node outputs, pseudo-values and cumulative log-gates by root-to-node replay.

    Returns o [T,H,dv], U [T,H,dv], G [T,H] (fp64).
    """
    ST0 = np.asarray(ST0, dtype=np.float64)
    B, H, dk, dv = ST0.shape
    parent = np.asarray(parent)
    cu_nodes = np.asarray(cu_nodes)
    _check_tree(parent, cu_nodes)
    T = int(cu_nodes[-1])
    o = np.zeros((T, H, dv))
    U = np.zeros((T, H, dv))
    G = np.zeros((T, H))
    for r in range(B):
        t0, t1 = int(cu_nodes[r]), int(cu_nodes[r + 1])
        par_r = parent[t0:t1]
        for h in range(H):
            for t in range(t1 - t0):
                S = ST0[r, h].T.copy()
                Gsum = 0.0
                u = None
                for j in _root_path(par_r, t):
                    a = float(np.exp(g[t0 + j, h]))
                    Gsum += float(g[t0 + j, h])
                    S, u = rule_step(S, a, float(beta[t0 + j, h]), k[t0 + j, h], v[t0 + j, h])
                o[t0 + t, h] = S @ q[t0 + t, h]
                U[t0 + t, h] = u
                G[t0 + t, h] = Gsum
    return o, U, G


def commit(ST0, k, v, beta, g, parent, cu_nodes, path, path_len):
    """State after replaying each request's accepted path (empty path keeps S_0). [B,H,dk,dv]."""
    ST0 = np.asarray(ST0, dtype=np.float64)
    B, H, dk, dv = ST0.shape
    _check_tree(parent, cu_nodes)
    _check_path(parent, cu_nodes, np.asarray(path), path_len)
    out = np.empty_like(ST0)
    for r in range(B):
        t0 = int(cu_nodes[r])
        for h in range(H):
            S = ST0[r, h].T.copy()
            for i in range(int(path_len[r])):
                j = t0 + int(path[r, i])
                S, _ = rule_step(S, float(np.exp(g[j, h])), float(beta[j, h]), k[j, h], v[j, h])
            out[r, h] = S.T
    return out


def accept_greedy(draft_tok, target_tok, parent, cu_nodes, max_path):
    """Greedy acceptance (GDN Tree-Scan abstract: device-side commitment of the accepted chain;
    TreeWY page, method section: outputs decide acceptance, then the accepted path is committed).

    Per request: start at node 0 (the root, always kept); at node x move to the lowest-indexed
    child c with draft_tok[c] == target_tok[x]; stop when no child matches or max_path nodes are
    taken. Returns (path [B, max_path] int32 padded with -1, path_len [B] int32, truncated [B] bool).
    Malformed trees (parent[t] outside [-1, t-1]) raise ValueError.
    """
    parent = np.asarray(parent)
    cu_nodes = np.asarray(cu_nodes)
    _check_tree(parent, cu_nodes)
    B = len(cu_nodes) - 1
    path = np.full((B, max_path), -1, dtype=np.int32)
    path_len = np.zeros(B, dtype=np.int32)
    truncated = np.zeros(B, dtype=bool)
    for r in range(B):
        t0, n = int(cu_nodes[r]), int(cu_nodes[r + 1] - cu_nodes[r])
        if n == 0:
            continue
        if max_path == 0:
            truncated[r] = True
            continue
        seq = [0]
        x = 0
        while True:
            match = [c for c in range(x + 1, n) if parent[t0 + c] == x and draft_tok[t0 + c] == target_tok[t0 + x]]
            if not match:
                break
            if len(seq) == max_path:
                truncated[r] = True
                break
            x = match[0]
            seq.append(x)
        path[r, :len(seq)] = seq
        path_len[r] = len(seq)
    return path, path_len, truncated
