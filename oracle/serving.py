"""Serving-layout forms of the oracle: state-pool slots, grouped query/key heads, a query scale
and gate pre-activations, written as the re-indexing and elementwise maps they are, in front
of the fp64 replay oracle.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only the tests, the smoke check and
the benchmark's CPU-baseline leg may import it; it shares no code with the CUDA kernels.

Definitions (the layout the ``*_ex`` entry points of the library accept):
  * request r reads and commits state ``pool[slot[r]]``; ``slot[r] == -1`` is a padding
    request (no outputs, no state change);
  * value head h reads query/key head ``h // (H // H_qk)``;
  * every query is multiplied by ``q_scale`` before the rule sees it (o = S (q_scale q));
  * with gate pre-activations, g = -exp(A_log[h]) softplus(a_raw + dt_bias[h]) and
    b = sigmoid(b_raw) replace the given g and beta. The TreeWY and GDN Tree-Scan pages do
    not print this parametrisation; it is the Gated DeltaNet one, taken here as the reading
    of "the gate / write strength computed just before the rule".
"""

from __future__ import annotations

import numpy as np

from . import commit as _commit
from . import verify as _verify


def softplus(x):
    """ln(1 + e^x) in fp64, without overflow for large x."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x):
    """1 / (1 + e^-x) in fp64, without overflow for very negative x."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def gate_beta(a_raw, b_raw, A_log, dt_bias):
    """g [T,H] and beta [T,H] from the pre-activations (A_log, dt_bias per head)."""
    a_raw = np.asarray(a_raw, dtype=np.float64)
    A_log = np.asarray(A_log, dtype=np.float64)
    dt_bias = np.asarray(dt_bias, dtype=np.float64)
    g = -np.exp(A_log)[None, :] * softplus(a_raw + dt_bias[None, :])
    return g, sigmoid(b_raw)


def expand_heads(x, H: int):
    """[T, H_qk, d] -> [T, H, d]: value head h takes head h // (H // H_qk)."""
    x = np.asarray(x, dtype=np.float64)
    H_qk = x.shape[1]
    if H % H_qk:
        raise ValueError("H must be a multiple of H_qk")
    return x[:, np.arange(H) // (H // H_qk), :]


def _states(pool, slot):
    slot = np.asarray(slot, dtype=np.int64)
    live = slot >= 0
    return np.asarray(pool, dtype=np.float64)[np.where(live, slot, 0)], live


def verify(pool, slot, q, k, v, beta, g, parent, cu_nodes, q_scale: float = 1.0, gates=None):
    """o, U, G [T,H,...] under the serving layout; rows of padding requests are NaN."""
    H = np.asarray(v).shape[1]
    if gates is not None:
        g, beta = gate_beta(*gates)
    ST0, live = _states(pool, slot)
    o, U, G = _verify(ST0, q_scale * expand_heads(q, H), expand_heads(k, H), v, beta, g, parent, cu_nodes)
    cu = np.asarray(cu_nodes)
    for r in np.flatnonzero(~live):
        o[cu[r]:cu[r + 1]] = np.nan
        U[cu[r]:cu[r + 1]] = np.nan
        G[cu[r]:cu[r + 1]] = np.nan
    return o, U, G


def commit(pool, slot, k, v, beta, g, parent, cu_nodes, path, path_len, gates=None):
    """The state pool after every live request's accepted path has been committed."""
    H = np.asarray(v).shape[1]
    if gates is not None:
        g, beta = gate_beta(*gates)
    ST0, live = _states(pool, slot)
    new = _commit(ST0, expand_heads(k, H), v, beta, g, parent, cu_nodes, path, path_len)
    out = np.array(pool, dtype=np.float64, copy=True)
    for r in np.flatnonzero(live):
        out[int(slot[r])] = new[r]
    return out
