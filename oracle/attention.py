"""Tree-bias attention oracle (fp64, plain loops over rows).

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; it shares no code with the CUDA kernels.

The attention layers of a hybrid model verify a draft tree in the same forward pass as its
Gated DeltaNet layers (GDN Tree-Scan abstract: tree-bias attention beside the recurrent-state
replay; for an attention-only model the verifier mainly needs an ancestry mask). Written out per
request r, query head h (key/value head h // (H_q / H_kv)) and draft node t:

    visible keys  = every key of the request's committed prefix
                    + the draft nodes on t's root-to-node path, t included
    o[t, h]       = sum_j softmax_j(scale * q[t, h] . k_j) v_j   over the visible keys j

Inputs are the library layouts widened to fp64: q [T, H_q, d], k, v [T, H_kv, d] (the draft
nodes' own keys and values), k_cache, v_cache [P_total, H_kv, d] with request r's prefix at rows
cu_prefix[r] .. cu_prefix[r+1]-1, parent [T] request-local (-1 = child of the prefix),
cu_nodes [B+1].
"""

from __future__ import annotations

import numpy as np


def _root_path(par, t):
    path = []
    while t >= 0:
        path.append(t)
        t = int(par[t])
    return path[::-1]


def tree_attention(q, k, v, k_cache, v_cache, cu_prefix, parent, cu_nodes, scale: float):
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    kc = np.asarray(k_cache, dtype=np.float64)
    vc = np.asarray(v_cache, dtype=np.float64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv:
        raise ValueError("H_q must be a multiple of H_kv")
    G = Hq // Hkv
    o = np.zeros((T, Hq, v.shape[2]))
    for r in range(len(cu_nodes) - 1):
        t0, t1 = int(cu_nodes[r]), int(cu_nodes[r + 1])
        p0, p1 = int(cu_prefix[r]), int(cu_prefix[r + 1])
        par = np.asarray(parent[t0:t1])
        for t in range(t1 - t0):
            if not (-1 <= par[t] < t):
                raise ValueError(f"request {r}: node {t} has parent {par[t]}")
            anc = [t0 + j for j in _root_path(par, t)]
            for h in range(Hq):
                g = h // G
                keys = np.concatenate([kc[p0:p1, g], k[anc, g]], axis=0)
                vals = np.concatenate([vc[p0:p1, g], v[anc, g]], axis=0)
                s = scale * (keys @ q[t0 + t, h])
                w = np.exp(s - s.max())
                o[t0 + t, h] = (w @ vals) / w.sum()
    return o
