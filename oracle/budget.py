"""Draft-budget oracle: which draft positions / tree nodes get verified.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; it shares no code with the CUDA kernels.

Two budgeting rules from the pages, written as plain step-by-step loops:

* ``topb`` - adaptive verification (DSpark adaptive-verification news item): each draft token
  has an estimated probability of passing verification; the probability that a request's
  sequence survives to position i is the product of those probabilities up to i; one global
  budget of B positions goes to the (request, position) pairs with the largest survival
  probabilities, so a late position of a confident request can outrank the first position of an
  unconfident one.
* ``grow_best_first`` - threshold best-first tree growth (TreeSpark page: the tree grows along
  the most promising branch first and stops once the value of the best remaining candidate
  drops below a threshold; a candidate's value is the survival product along its branch).

Survival products decide integers (which positions, which nodes), so they are formed in fp32,
multiplying along the path from the root in order - the precision the kernels use - and the
comparisons are exact. Ties are broken by the smaller (request, position) pair, and by the
smaller candidate index.
"""

from __future__ import annotations

import heapq

import numpy as np

F32 = np.float32


def _prob(x) -> np.float32:
    """An estimated probability: values outside [0, 1] (or NaN) count as 0 (never chosen)."""
    x = F32(x)
    return x if (x >= 0 and x <= 1) else F32(0)


def survival(p_accept) -> np.ndarray:
    """s[r, i] = p[r, 0] * p[r, 1] * ... * p[r, i] in fp32, multiplied left to right."""
    p = np.asarray(p_accept, dtype=np.float32)
    R, K = p.shape
    s = np.zeros((R, K), dtype=np.float32)
    for r in range(R):
        acc = F32(1)
        for i in range(K):
            acc = F32(acc * _prob(p[r, i]))
            s[r, i] = acc
    return s


def topb(p_accept, budget: int):
    """Top-B allocation of draft positions across requests.

    Returns (n_sel [R], survival [R, K], cu_nodes [R+1], parent [T]): request r verifies its
    first n_sel[r] draft positions, as a chain of 1 + n_sel[r] nodes (node 0 = the token the
    target already produced, then the chosen drafts), packed in request order.
    """
    s = survival(p_accept)
    R, K = s.shape
    items = [(-float(s[r, i]), r, i) for r in range(R) for i in range(K)]
    items.sort()
    n_sel = np.zeros(R, dtype=np.int32)
    for _, r, i in items[:max(0, min(int(budget), R * K))]:
        n_sel[r] += 1
    cu = np.zeros(R + 1, dtype=np.int32)
    parent = []
    for r in range(R):
        n = 1 + int(n_sel[r])
        cu[r + 1] = cu[r] + n
        parent.extend(range(-1, n - 1))
    return n_sel, s, cu, np.asarray(parent, dtype=np.int32)


def candidate_count(fanout: int, depth: int) -> int:
    """Nodes of the complete fanout-ary candidate tree of the given depth (root included)."""
    return sum(fanout ** l for l in range(depth + 1))


def grow_best_first(p_edge, fanout: int, depth: int, threshold: float, max_nodes: int):
    """Threshold best-first growth over a complete candidate tree, one request at a time.

    Candidates are numbered breadth-first: 0 is the root (the token the target already
    produced, value 1, always taken), the children of c are fanout*c + 1 .. fanout*c + fanout,
    and p_edge[r, c] is the estimated probability that candidate c is accepted given its
    parent. Starting from the root, repeatedly take the frontier candidate of largest value
    (value = product of p_edge along its branch; ties -> smaller index); stop when it is below
    ``threshold`` or ``max_nodes`` nodes are taken; a taken candidate's children join the
    frontier. Returns per request the taken candidates in the order taken, their request-local
    parent indices, and values - as padded [R, max_nodes] arrays (-1 / 0 past n) plus
    n_nodes [R], and the packed (cu_nodes, parent) of the resulting ragged batch.
    """
    p = np.asarray(p_edge, dtype=np.float32)
    R, C = p.shape
    if C != candidate_count(fanout, depth):
        raise ValueError("p_edge must have one column per candidate")
    thr = F32(threshold)
    cand = np.full((R, max_nodes), -1, dtype=np.int32)
    par = np.full((R, max_nodes), -1, dtype=np.int32)
    val = np.zeros((R, max_nodes), dtype=np.float32)
    n_nodes = np.zeros(R, dtype=np.int32)
    for r in range(R):
        if max_nodes < 1:
            continue
        taken_at = {}  # candidate -> output index
        frontier = [(-1.0, 0, F32(1))]  # (-value, candidate, value)
        n = 0
        while frontier and n < max_nodes:
            negv, c, v = heapq.heappop(frontier)
            if c != 0 and not (v >= thr):
                break  # the best remaining candidate is below the threshold
            cand[r, n], val[r, n] = c, v
            par[r, n] = -1 if c == 0 else taken_at[(c - 1) // fanout]
            taken_at[c] = n
            n += 1
            for ch in range(fanout * c + 1, fanout * c + fanout + 1):
                if ch < C:
                    cv = F32(v * _prob(p[r, ch]))
                    heapq.heappush(frontier, (-float(cv), ch, cv))
        n_nodes[r] = n
    cu = np.zeros(R + 1, dtype=np.int32)
    cu[1:] = np.cumsum(n_nodes)
    parent = np.concatenate([par[r, :n_nodes[r]] for r in range(R)]) if R else np.zeros(0, np.int32)
    return {"cand": cand, "parent_local": par, "value": val, "n_nodes": n_nodes, "cu_nodes": cu,
            "parent": parent.astype(np.int32)}
