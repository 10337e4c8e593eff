"""Seeded synthetic inputs for draft-tree verification of a Gated DeltaNet layer.

This module only *draws* inputs. It holds none of the method's arithmetic
(no recurrence, no solve, no commit), so the CPU oracle and the CUDA path can
both be fed from it without sharing any computation.

Workload presets (``make_config(i)``; sizes, shapes and distributions of the synthetic
workloads the TreeWY and GDN Tree-Scan pages motivate):

* 0 - one request, one head, d=32, a chain of 3 draft nodes, accepted path = first 2.
* 1 - depth-3 chain (bonus + 3 drafts = 4 nodes), 256 requests, 32 heads, d=128
  (the "depth-3 chain" setting of the TreeWY page, experiments section).
* 2 - the 6-node root-branch tree of the GDN Tree-Scan abstract (root with 3
  children, 2 of them with one child each), batch 1 or 64, 48 heads.
* 3 - ragged random trees of 16..64 nodes (fanout 1..4, depth <= 8), batch 128.
* 4 - 32-node random trees (fanout 1..3, depth <= 6), gate a ~ U(0.85, 1),
  batch 1..512, 32 heads, one independent input set per GDN layer.

Value recipe (all presets): state S ~ N(0, 0.1^2) in fp32; q, k ~ N(0, 1) drawn in
fp32, L2-normalised in fp32, then rounded to bf16 (round-to-nearest-even);
v ~ N(0, 1) rounded to bf16; beta ~ U(0, 1) fp32; gate a = exp(-0.1*softplus(x)),
x ~ N(0, 1), passed as the natural log g = ln a (fp32).

Layouts (the library's HBM layouts):
  ST   [B, H, d_k, d_v] fp32   (the state S is d_v x d_k; it is stored transposed)
  q, k [T, H, d_k]      bf16   (stored here as uint16 bit patterns)
  v    [T, H, d_v]      bf16
  beta, g [T, H]        fp32
  parent [T] int32, request-local, -1 = child of the committed state, parent[t] < t
  cu_nodes [B + 1] int32 node offsets
  path [B, max_path] int32 (request-local node ids, root -> node, padded with -1)
  path_len [B] int32
"""

from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np

MAX_NODES = 64

# ---------------------------------------------------------------------------
# bf16 helpers (bit-level, round to nearest even)
# ---------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even) and return the 16-bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounding_bias = 0x7FFF + ((u >> 16) & 1)
    out = ((u + rounding_bias) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# tree shapes
# ---------------------------------------------------------------------------


def chain_parents(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def root_branch_parents() -> np.ndarray:
    """Six-node root-branch tree: root 0 with children 1, 2, 3; 1 -> 4, 2 -> 5."""
    return np.array([-1, 0, 0, 0, 1, 2], dtype=np.int32)


def random_tree_parents(rng: np.random.Generator, n: int, fanout_max: int, depth_max: int) -> np.ndarray:
    """Breadth-first random tree of exactly ``n`` nodes, parent-before-child order.

    A popped node of depth < depth_max gets f ~ U{1..fanout_max} children, capped by the
    remaining budget. If the queue runs dry before ``n`` nodes exist, one child is added to
    the earliest node that still has depth < depth_max and fewer than fanout_max children.
    Depth counts edges from the root (root depth 0).
    """
    if n < 1:
        return np.zeros(0, dtype=np.int32)
    parent = [-1]
    depth = [0]
    nchild = [0]
    queue = deque([0])

    def add(p: int) -> None:
        parent.append(p)
        depth.append(depth[p] + 1)
        nchild.append(0)
        nchild[p] += 1
        queue.append(len(parent) - 1)

    while len(parent) < n:
        if queue:
            x = queue.popleft()
            if depth[x] >= depth_max:
                continue
            f = int(rng.integers(1, fanout_max + 1))
            f = min(f, fanout_max - nchild[x], n - len(parent))
            for _ in range(f):
                add(x)
        else:
            cand = [i for i in range(len(parent)) if depth[i] < depth_max and nchild[i] < fanout_max]
            if not cand:
                raise ValueError("tree limits too tight for the requested node count")
            add(cand[0])
    return np.asarray(parent, dtype=np.int32)


def random_topological_relabel(rng: np.random.Generator, parent: np.ndarray):
    """Relabel a parent-before-child tree by a uniformly chosen topological order.

    Returns (new_parent, perm) with perm[new_index] = old_index.
    """
    n = len(parent)
    children = [[] for _ in range(n)]
    avail = []
    for t in range(n):
        if parent[t] < 0:
            avail.append(t)
        else:
            children[parent[t]].append(t)
    order = []
    while avail:
        i = int(rng.integers(len(avail)))
        x = avail.pop(i)
        order.append(x)
        avail.extend(children[x])
    perm = np.asarray(order, dtype=np.int64)
    inv = np.empty(n, dtype=np.int64)
    inv[perm] = np.arange(n)
    new_parent = np.array([-1 if parent[o] < 0 else inv[parent[o]] for o in perm], dtype=np.int32)
    return new_parent, perm


def root_path(parent: np.ndarray, node: int) -> list[int]:
    """Request-local node ids from the root down to ``node`` (inclusive)."""
    out = []
    x = int(node)
    while x >= 0:
        out.append(x)
        x = int(parent[x])
    return out[::-1]


def leaves(parent: np.ndarray) -> list[int]:
    has_child = np.zeros(len(parent), dtype=bool)
    for p in parent:
        if p >= 0:
            has_child[p] = True
    return [i for i in range(len(parent)) if not has_child[i]]


def greedy_walk_path(rng: np.random.Generator, parent: np.ndarray) -> list[int]:
    """Start at root 0 (always taken); at each node choose uniformly among {stop} + children."""
    children = [[] for _ in range(len(parent))]
    for t, p in enumerate(parent):
        if p >= 0:
            children[p].append(t)
    path = [0]
    x = 0
    while children[x]:
        choice = int(rng.integers(len(children[x]) + 1))
        if choice == len(children[x]):
            break
        x = children[x][choice]
        path.append(x)
    return path


def leaf_prefix_path(rng: np.random.Generator, parent: np.ndarray) -> list[int]:
    """Uniform leaf, then a prefix of its root path with length uniform in 1..len."""
    lv = leaves(parent)
    leaf = lv[int(rng.integers(len(lv)))]
    full = root_path(parent, leaf)
    m = int(rng.integers(1, len(full) + 1))
    return full[:m]


# ---------------------------------------------------------------------------
# batches
# ---------------------------------------------------------------------------


@dataclass
class TreeBatch:
    """One layer's verify + commit inputs, host-side (numpy)."""

    B: int
    H: int
    dk: int
    dv: int
    parent: np.ndarray  # [T] int32
    cu_nodes: np.ndarray  # [B+1] int32
    path: np.ndarray  # [B, max_path] int32, -1 padded
    path_len: np.ndarray  # [B] int32
    ST0: np.ndarray  # [B, H, dk, dv] fp32
    q: np.ndarray  # [T, H, dk] uint16 (bf16 bits)
    k: np.ndarray  # [T, H, dk] uint16
    v: np.ndarray  # [T, H, dv] uint16
    beta: np.ndarray  # [T, H] fp32
    g: np.ndarray  # [T, H] fp32 (natural log of the gate a)
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.cu_nodes[-1])

    @property
    def max_nodes(self) -> int:
        if self.B == 0:
            return 0
        return int(np.max(np.diff(self.cu_nodes)))

    @property
    def max_path(self) -> int:
        return int(self.path.shape[1])

    def n_nodes(self, r: int) -> int:
        return int(self.cu_nodes[r + 1] - self.cu_nodes[r])

    def request_parent(self, r: int) -> np.ndarray:
        return self.parent[self.cu_nodes[r]:self.cu_nodes[r + 1]]

    def q_f32(self):
        return bf16_bits_to_f32(self.q)

    def k_f32(self):
        return bf16_bits_to_f32(self.k)

    def v_f32(self):
        return bf16_bits_to_f32(self.v)


def _normalised_bf16(rng, shape, dtype=np.float32):
    x = rng.standard_normal(shape, dtype=np.float32)
    nrm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32), dtype=np.float32)
    x = (x / nrm).astype(np.float32)
    return f32_to_bf16_bits(x)


def gate_softplus(rng, shape, scale=0.1) -> np.ndarray:
    """g = ln a with a = exp(-scale * softplus(x)), x ~ N(0, 1)."""
    x = rng.standard_normal(shape)
    return (-scale * np.logaddexp(0.0, x)).astype(np.float32)


def gate_uniform(rng, shape, lo=0.85, hi=1.0) -> np.ndarray:
    """g = ln a with a ~ U(lo, hi)."""
    a = rng.uniform(lo, hi, size=shape)
    return np.log(a).astype(np.float32)


def build_batch(rng: np.random.Generator, parents: list, paths: list, H: int, dk: int, dv: int,
                gate: str = "softplus", state_std: float = 0.1, name: str = "") -> TreeBatch:
    """Draw one layer's tensors for the given per-request trees and accepted paths."""
    B = len(parents)
    sizes = [len(p) for p in parents]
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(sizes)
    T = int(cu[-1])
    parent = np.concatenate([np.asarray(p, dtype=np.int32) for p in parents]) if T else np.zeros(0, np.int32)
    max_path = max([len(p) for p in paths] + [1])
    path = np.full((B, max_path), -1, dtype=np.int32)
    path_len = np.zeros(B, dtype=np.int32)
    for r, p in enumerate(paths):
        path[r, :len(p)] = p
        path_len[r] = len(p)
    ST0 = (rng.standard_normal((B, H, dk, dv), dtype=np.float32) * np.float32(state_std)).astype(np.float32)
    q = _normalised_bf16(rng, (T, H, dk))
    k = _normalised_bf16(rng, (T, H, dk))
    v = f32_to_bf16_bits(rng.standard_normal((T, H, dv), dtype=np.float32))
    beta = rng.uniform(0.0, 1.0, size=(T, H)).astype(np.float32)
    if gate == "softplus":
        g = gate_softplus(rng, (T, H))
    elif gate == "uniform":
        g = gate_uniform(rng, (T, H))
    else:
        raise ValueError(gate)
    return TreeBatch(B=B, H=H, dk=dk, dv=dv, parent=parent, cu_nodes=cu, path=path, path_len=path_len,
                     ST0=ST0, q=q, k=k, v=v, beta=beta, g=g, name=name)


CONFIG_BATCHES = {0: (1,), 1: (256,), 2: (1, 64), 3: (128,), 4: (1, 8, 32, 128, 256, 512)}
CONFIG_LAYERS = {0: 1, 1: 1, 2: 1, 3: 1, 4: 48}


def make_config(idx: int, batch: int | None = None, layer: int = 0, heads: int | None = None) -> TreeBatch:
    """Build one layer of workload preset ``idx`` (0..4, see the module docstring).

    ``batch`` picks one of the preset's batch sizes (default: the largest listed);
    ``heads`` may shrink the head count for quick tests (same per-head distributions).
    """
    if batch is None:
        batch = CONFIG_BATCHES[idx][-1]
    ss = np.random.SeedSequence([idx, batch, layer])
    rng = np.random.default_rng(ss)
    if idx == 0:
        parents = [chain_parents(3)]
        paths = [[0, 1]]
        return build_batch(rng, parents, paths, H=heads or 1, dk=32, dv=32, name="chain3_d32")
    if idx == 1:
        parents, paths = [], []
        for _ in range(batch):
            parents.append(chain_parents(4))
            L = int(rng.integers(0, 4))  # accepted drafts after the always-committed bonus node
            paths.append(list(range(L + 1)))
        return build_batch(rng, parents, paths, H=heads or 32, dk=128, dv=128,
                           name=f"chain4_B{batch}")
    if idx == 2:
        parents, paths = [], []
        for _ in range(batch):
            p = root_branch_parents()
            parents.append(p)
            paths.append(greedy_walk_path(rng, p))
        return build_batch(rng, parents, paths, H=heads or 48, dk=128, dv=128,
                           name=f"rootbranch6_B{batch}")
    if idx == 3:
        parents, paths = [], []
        for _ in range(batch):
            n = int(rng.integers(16, 65))
            p = random_tree_parents(rng, n, fanout_max=4, depth_max=8)
            parents.append(p)
            paths.append(leaf_prefix_path(rng, p))
        return build_batch(rng, parents, paths, H=heads or 32, dk=128, dv=128,
                           name=f"ragged16to64_B{batch}")
    if idx == 4:
        parents, paths = [], []
        for _ in range(batch):
            p = random_tree_parents(rng, 32, fanout_max=3, depth_max=6)
            parents.append(p)
            paths.append(leaf_prefix_path(rng, p))
        return build_batch(rng, parents, paths, H=heads or 32, dk=128, dv=128, gate="uniform",
                           name=f"tree32_B{batch}_layer{layer}")
    raise ValueError(f"unknown config {idx}")


def make_random_batch(seed: int, B: int, H: int, d: int, n_range=(1, 16), fanout_max=3, depth_max=6,
                      shuffle_order: bool = True, gate: str = "softplus", empty_every: int = 0) -> TreeBatch:
    """Small random ragged batch for tests (random topological orders, optional empty requests)."""
    rng = np.random.default_rng(seed)
    parents, paths = [], []
    for r in range(B):
        if empty_every and r % empty_every == empty_every - 1:
            parents.append(np.zeros(0, np.int32))
            paths.append([])
            continue
        n = int(rng.integers(n_range[0], n_range[1] + 1))
        p = random_tree_parents(rng, n, fanout_max=fanout_max, depth_max=depth_max)
        if shuffle_order:
            p, _ = random_topological_relabel(rng, p)
        parents.append(p)
        lv = leaves(p)
        full = root_path(p, lv[int(rng.integers(len(lv)))])
        paths.append(full[:int(rng.integers(0, len(full) + 1))])
    return build_batch(rng, parents, paths, H=H, dk=d, dv=d, gate=gate, name=f"random_seed{seed}")


@dataclass
class ServingInputs:
    """Serving-layout inputs that go with a TreeBatch (see ``make_serving_batch``)."""

    pool: np.ndarray  # [n_slots, H, dk, dv] fp32 state pool
    slot: np.ndarray  # [B] int32 state slot per request, -1 = padding request
    H_qk: int  # query/key heads (H is a multiple)
    q: np.ndarray  # [T, H_qk, dk] uint16 (bf16 bits)
    k: np.ndarray  # [T, H_qk, dk] uint16
    q_scale: float
    a_raw: np.ndarray  # [T, H] fp32 gate pre-activation
    b_raw: np.ndarray  # [T, H] fp32 write-strength pre-activation
    A_log: np.ndarray  # [H] fp32
    dt_bias: np.ndarray  # [H] fp32

    @property
    def gates(self):
        return self.a_raw, self.b_raw, self.A_log, self.dt_bias


def make_serving_batch(seed: int, B: int, H: int, H_qk: int, d: int, n_range=(1, 16), n_slots: int | None = None,
                       pad_every: int = 0, q_scale: float | None = None, **tree_kw):
    """A random ragged batch laid out as a serving engine holds it: states in a pool larger than
    the batch (distinct random slots, every ``pad_every``-th request a -1 padding slot), q and k
    with H_qk heads, a query scale (default d^-1/2), and gate pre-activations
    a_raw ~ N(0, 1), b_raw ~ N(0, 1), A_log = ln U(1, 16), dt_bias ~ U(-7, -2) (per-step decays
    of roughly 0.8 .. 1 once mapped through the gate). Returns (TreeBatch, ServingInputs); the
    TreeBatch's own q, k and ST0 are not used by the serving layout."""
    tb = make_random_batch(seed=seed, B=B, H=H, d=d, n_range=n_range, **tree_kw)
    rng = np.random.default_rng([seed, 0x5e])
    n_slots = n_slots if n_slots is not None else 2 * B + 3
    if n_slots < B:
        raise ValueError("the pool must hold a state per request")
    slot = rng.permutation(n_slots)[:B].astype(np.int32)
    if pad_every:
        slot[pad_every - 1::pad_every] = -1
    pool = (rng.standard_normal((n_slots, H, d, d), dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    T = tb.T
    sv = ServingInputs(
        pool=pool, slot=slot, H_qk=H_qk,
        q=_normalised_bf16(rng, (T, H_qk, d)), k=_normalised_bf16(rng, (T, H_qk, d)),
        q_scale=float(d ** -0.5) if q_scale is None else float(q_scale),
        a_raw=rng.standard_normal((T, H), dtype=np.float32),
        b_raw=rng.standard_normal((T, H), dtype=np.float32),
        A_log=np.log(rng.uniform(1.0, 16.0, size=H)).astype(np.float32),
        dt_bias=rng.uniform(-7.0, -2.0, size=H).astype(np.float32))
    return tb, sv


def draw_tokens(rng: np.random.Generator, parent: np.ndarray, cu_nodes: np.ndarray, vocab: int = 50,
                p_match: float = 0.7):
    """Synthetic draft / target tokens for greedy acceptance tests.

    draft_tok[t] is uniform over the vocabulary. target_tok[x] (the target's greedy token after
    node x) equals the draft token of one of x's children, chosen uniformly, with probability
    p_match, and is uniform otherwise (a leaf always gets a uniform token).
    """
    T = int(cu_nodes[-1])
    draft = rng.integers(0, vocab, size=T).astype(np.int32)
    target = rng.integers(0, vocab, size=T).astype(np.int32)
    for r in range(len(cu_nodes) - 1):
        t0, t1 = int(cu_nodes[r]), int(cu_nodes[r + 1])
        children = [[] for _ in range(t1 - t0)]
        for t in range(t0, t1):
            p = int(parent[t])
            if p >= 0:
                children[p].append(t - t0)
        for x in range(t1 - t0):
            if children[x] and rng.random() < p_match:
                target[t0 + x] = draft[t0 + children[x][int(rng.integers(len(children[x])))]]
    return draft, target


def draw_acceptance(rng: np.random.Generator, R: int, K: int) -> np.ndarray:
    """Estimated per-position acceptance probabilities [R, K] fp32 for draft budgeting.

    Request r has a confidence c_r ~ U(0.6, 1); position i's probability is c_r * 0.9^i plus
    N(0, 0.02) noise, clipped to [0, 1]. With K = 7 the first position is accepted ~80 % of the
    time and the seventh survives ~3 % of the time on average, the spread the DSpark news item
    reports (above 70 % for the first of seven drafts, below 10 % for the last).
    """
    c = rng.uniform(0.6, 1.0, size=(R, 1))
    p = c * 0.9 ** np.arange(K)[None, :] + rng.normal(0.0, 0.02, size=(R, K))
    return np.clip(p, 0.0, 1.0).astype(np.float32)


def draw_edge_probs(rng: np.random.Generator, R: int, fanout: int, depth: int, alpha: float = 0.6) -> np.ndarray:
    """Per-candidate acceptance probabilities [R, C] fp32 over a complete fanout-ary candidate
    tree (breadth-first numbering, C = sum_l fanout^l, column 0 = the root, set to 1).

    The children of each candidate share one Dirichlet(alpha) draw over fanout + 1 outcomes
    (the last: no child accepted), sorted so that the first child is the most likely, as the
    ranked alternatives of a drafter would be.
    """
    C = sum(fanout ** l for l in range(depth + 1))
    p = np.ones((R, C), dtype=np.float32)
    n_internal = (C - 1) // fanout  # candidates with children
    w = rng.dirichlet(np.full(fanout + 1, alpha), size=(R, n_internal))[:, :, :fanout]
    w = -np.sort(-w, axis=2)
    p[:, 1:] = w.reshape(R, n_internal * fanout).astype(np.float32)
    return p


@dataclass
class AttentionBatch:
    """Inputs of one tree-bias attention layer (see ``make_attention_batch``)."""

    B: int
    Hq: int
    Hkv: int
    d: int
    parent: np.ndarray     # [T] int32
    cu_nodes: np.ndarray   # [B+1] int32
    cu_prefix: np.ndarray  # [B+1] int32
    q: np.ndarray          # [T, Hq, d] uint16 (bf16 bits)
    k: np.ndarray          # [T, Hkv, d] uint16
    v: np.ndarray          # [T, Hkv, d] uint16
    k_cache: np.ndarray    # [P_total, Hkv, d] uint16
    v_cache: np.ndarray    # [P_total, Hkv, d] uint16
    scale: float

    @property
    def T(self) -> int:
        return int(self.cu_nodes[-1])

    @property
    def P(self) -> int:
        return int(self.cu_prefix[-1])

    @property
    def max_nodes(self) -> int:
        return int(np.max(np.diff(self.cu_nodes))) if self.B else 0

    @property
    def max_prefix(self) -> int:
        return int(np.max(np.diff(self.cu_prefix))) if self.B else 0


def make_attention_batch(seed: int, B: int, Hq: int, Hkv: int, d: int, prefix_range=(0, 512), parents=None,
                         n_range=(1, 16), fanout_max=3, depth_max=6) -> AttentionBatch:
    """Tree-bias attention inputs: a committed key/value prefix per request, of length uniform
    in ``prefix_range``, and a draft tree per request (``parents``, or random trees as in
    ``make_random_batch``). q, k, v and the caches are N(0, 1) rounded to bf16; the score scale
    is d^-1/2."""
    rng = np.random.default_rng([seed, 0xa7])
    if parents is None:
        parents = []
        for _ in range(B):
            n = int(rng.integers(n_range[0], n_range[1] + 1))
            parents.append(random_tree_parents(rng, n, fanout_max=fanout_max, depth_max=depth_max))
    sizes = [len(p) for p in parents]
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(sizes)
    plen = rng.integers(prefix_range[0], prefix_range[1] + 1, size=B)
    cp = np.zeros(B + 1, dtype=np.int32)
    cp[1:] = np.cumsum(plen)
    T, P = int(cu[-1]), int(cp[-1])
    bf = lambda *shape: f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    parent = np.concatenate([np.asarray(p, np.int32) for p in parents]) if T else np.zeros(0, np.int32)
    return AttentionBatch(B=B, Hq=Hq, Hkv=Hkv, d=d, parent=parent, cu_nodes=cu, cu_prefix=cp,
                          q=bf(T, Hq, d), k=bf(T, Hkv, d), v=bf(T, Hkv, d), k_cache=bf(P, Hkv, d),
                          v_cache=bf(P, Hkv, d), scale=float(d ** -0.5))


# ---------------------------------------------------------------------------
# the same presets drawn on a CUDA device (for timing many large layers)
# ---------------------------------------------------------------------------

@dataclass
class TreeShape:
    """The integer part of one preset layer: trees and accepted paths, no values."""

    B: int
    H: int
    dk: int
    dv: int
    parent: np.ndarray
    cu_nodes: np.ndarray
    path: np.ndarray
    path_len: np.ndarray
    gate: str
    name: str = ""

    @property
    def T(self) -> int:
        return int(self.cu_nodes[-1])

    @property
    def max_nodes(self) -> int:
        return int(np.max(np.diff(self.cu_nodes))) if self.B else 0

    @property
    def max_path(self) -> int:
        return int(self.path.shape[1])


def config_shape(idx: int, batch: int | None = None, layer: int = 0) -> TreeShape:
    """The trees and accepted paths of ``make_config(idx, batch, layer)`` (the same draws from
    the same seed), without drawing the layer's values."""
    if batch is None:
        batch = CONFIG_BATCHES[idx][-1]
    rng = np.random.default_rng(np.random.SeedSequence([idx, batch, layer]))
    H, d, gate = 32, 128, "softplus"
    parents, paths = [], []
    if idx == 0:
        parents, paths, H, d = [chain_parents(3)], [[0, 1]], 1, 32
    elif idx == 1:
        for _ in range(batch):
            parents.append(chain_parents(4))
            paths.append(list(range(int(rng.integers(0, 4)) + 1)))
    elif idx == 2:
        H = 48
        for _ in range(batch):
            p = root_branch_parents()
            parents.append(p)
            paths.append(greedy_walk_path(rng, p))
    elif idx == 3:
        for _ in range(batch):
            p = random_tree_parents(rng, int(rng.integers(16, 65)), fanout_max=4, depth_max=8)
            parents.append(p)
            paths.append(leaf_prefix_path(rng, p))
    elif idx == 4:
        gate = "uniform"
        for _ in range(batch):
            p = random_tree_parents(rng, 32, fanout_max=3, depth_max=6)
            parents.append(p)
            paths.append(leaf_prefix_path(rng, p))
    else:
        raise ValueError(f"unknown config {idx}")
    B = len(parents)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum([len(p) for p in parents])
    max_path = max([len(p) for p in paths] + [1])
    path = np.full((B, max_path), -1, dtype=np.int32)
    path_len = np.zeros(B, dtype=np.int32)
    for r, p in enumerate(paths):
        path[r, :len(p)] = p
        path_len[r] = len(p)
    parent = np.concatenate([np.asarray(p, dtype=np.int32) for p in parents])
    return TreeShape(B=B, H=H, dk=d, dv=d, parent=parent, cu_nodes=cu, path=path, path_len=path_len, gate=gate,
                     name=f"config{idx}_B{batch}_layer{layer}")


def draw_values_device(shape: TreeShape, seed: int, device) -> dict:
    """One layer's values for ``shape`` drawn on ``device`` with the presets' value recipe
    (torch's seeded generator instead of numpy's): S ~ N(0, 0.1^2) fp32; q, k ~ N(0, 1)
    L2-normalised in fp32 then rounded to bf16; v ~ N(0, 1) in bf16; beta ~ U(0, 1);
    g = ln a with a = exp(-0.1 softplus(x)), x ~ N(0, 1), or a ~ U(0.85, 1)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    T, H, dk, dv = shape.T, shape.H, shape.dk, shape.dv
    f32 = dict(dtype=torch.float32, device=device, generator=gen)

    def unit_rows(*s):
        x = torch.randn(*s, **f32)
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)

    out = {"ST": torch.randn(shape.B, H, dk, dv, **f32) * 0.1, "q": unit_rows(T, H, dk), "k": unit_rows(T, H, dk),
           "v": torch.randn(T, H, dv, **f32).to(torch.bfloat16), "beta": torch.rand(T, H, **f32)}
    if shape.gate == "uniform":
        out["g"] = torch.log(0.85 + 0.15 * torch.rand(T, H, **f32))
    else:
        out["g"] = -0.1 * torch.nn.functional.softplus(torch.randn(T, H, **f32))
    for key, arr in (("parent", shape.parent), ("cu_nodes", shape.cu_nodes), ("path", shape.path),
                     ("path_len", shape.path_len)):
        out[key] = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32)).to(device)
    return out
