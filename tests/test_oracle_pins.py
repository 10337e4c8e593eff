"""Pins for the CPU oracle (both the C replay and its NumPy twin).

The oracle replays the gated delta rule along every root-to-node path. These tests tie it
to facts fixed outside the oracle itself, chosen so that a plausible slip anywhere in it -
a dropped term, a wrong sign, a transposed state, a gate on the wrong factor, a wrong
ancestor set - fails at least one of them (``test_planted_mistakes_are_caught`` plants each
such slip in the NumPy twin and checks that):

* a hand-worked d=2 tree (``tests/golden/worked_example_d2.txt``, exact fractions);
* closed forms of the rule: beta = 0 (no write: pure decay by the path's gate product),
  delta-rule erasure (beta = 1, |k| = 1, q = k  =>  o = v), a single node on a zero state,
  and orthonormal keys, where the replay collapses to a sum over the root-to-node path;
* invariants: joint linearity in (S_0, v), chain = token-by-token sequential decode
  (GDN Tree-Scan abstract), branch extraction (a node's output only depends on its own
  root-to-node path - TreeWY page, method section), relabelling by another topological
  order, commit state applied to q reproduces the accepted node's output;
* brute-force store-all stepping from each parent's stored state (the storeall baseline
  the TreeWY page describes under its comparison with prior methods);
* the tree-structured WY identity in fp64 (one triangular system, TreeWY page, method
  section) - a check of the derivation the CUDA path uses, not of the CUDA path.
"""

import math
import os

import numpy as np
import pytest

import oracle
from oracle import replay
from gated_deltanet_tree_03_b300 import workloads as W

IMPLS = ["c", "numpy"]


# ---------------------------------------------------------------------------
# uniform access to both oracle implementations
# ---------------------------------------------------------------------------

def run_verify(impl, ST0, q, k, v, beta, g, parent, cu):
    if impl == "c":
        return oracle.verify(ST0, q, k, v, beta, g, parent, cu)
    return replay.verify(ST0, q, k, v, beta, g, parent, cu)


def run_commit(impl, ST0, k, v, beta, g, parent, cu, path, path_len):
    if impl == "c":
        return oracle.commit(ST0, k, v, beta, g, parent, cu, path, path_len)
    return replay.commit(ST0, k, v, beta, g, parent, cu, np.asarray(path), path_len)


def ancestors_plus(parent_r, t):
    """Root-to-node node list by walking parents (brute force, independent of the oracle)."""
    out = []
    x = t
    while x >= 0:
        out.append(x)
        x = int(parent_r[x])
    return out[::-1]


def rand_inputs(rng, parents, H, dk, dv, paths=None, unit_keys=True):
    sizes = [len(p) for p in parents]
    cu = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    T = int(cu[-1])
    parent = np.concatenate(parents).astype(np.int32)
    B = len(parents)
    ST0 = rng.normal(0, 0.3, (B, H, dk, dv))
    q = rng.normal(size=(T, H, dk))
    k = rng.normal(size=(T, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.normal(size=(T, H, dv))
    beta = rng.uniform(0, 1, (T, H))
    g = -0.3 * np.logaddexp(0, rng.normal(size=(T, H)))
    if paths is None:
        paths = []
        for p in parents:
            lv = W.leaves(np.asarray(p))
            full = W.root_path(np.asarray(p), lv[int(rng.integers(len(lv)))])
            paths.append(full[:int(rng.integers(0, len(full) + 1))])
    max_path = max([len(p) for p in paths] + [1])
    path = np.full((B, max_path), -1, np.int32)
    plen = np.zeros(B, np.int32)
    for r, p in enumerate(paths):
        path[r, :len(p)] = p
        plen[r] = len(p)
    return dict(ST0=ST0, q=q, k=k, v=v, beta=beta, g=g, parent=parent, cu=cu, path=path, plen=plen)


def random_parents(rng, n, shuffle=True, fanout=3, depth=5):
    p = W.random_tree_parents(rng, n, fanout_max=fanout, depth_max=depth)
    if shuffle:
        p, _ = W.random_topological_relabel(rng, p)
    return p


def verify_of(impl, x):
    return run_verify(impl, x["ST0"], x["q"], x["k"], x["v"], x["beta"], x["g"], x["parent"], x["cu"])


def commit_of(impl, x):
    return run_commit(impl, x["ST0"], x["k"], x["v"], x["beta"], x["g"], x["parent"], x["cu"],
                      x["path"], x["plen"])


# ---------------------------------------------------------------------------
# pins (each is a plain function so the planted-mistake test can rerun them)
# ---------------------------------------------------------------------------

def load_worked_example():
    path = os.path.join(os.path.dirname(__file__), "golden", "worked_example_d2.txt")
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = np.array([float(x) for x in rest.split()])
    return vals


def pin_worked_example(impl):
    ex = load_worked_example()
    parent = ex["parent"].astype(np.int32)
    cu = np.array([0, 3], np.int32)
    ST0 = ex["ST0"].reshape(1, 1, 2, 2)
    q = ex["q"].reshape(3, 1, 2)
    k = ex["k"].reshape(3, 1, 2)
    v = ex["v"].reshape(3, 1, 2)
    beta = ex["beta"].reshape(3, 1)
    g = np.log(ex["a"]).reshape(3, 1)
    o, U, G = run_verify(impl, ST0, q, k, v, beta, g, parent, cu)
    np.testing.assert_allclose(o.reshape(3, 2), ex["o"].reshape(3, 2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(U.reshape(3, 2), ex["U"].reshape(3, 2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(G.reshape(3), ex["G"], rtol=0, atol=1e-12)
    for name, p in [("commit_path_0_2", [0, 2]), ("commit_path_0_1", [0, 1]), ("commit_path_empty", [])]:
        path = np.full((1, 2), -1, np.int32)
        path[0, :len(p)] = p
        ST = run_commit(impl, ST0, k, v, beta, g, parent, cu, path, np.array([len(p)], np.int32))
        np.testing.assert_allclose(ST.reshape(4), ex[name], rtol=0, atol=1e-12)


def pin_no_write(impl, seed=1):
    rng = np.random.default_rng(seed)
    parents = [random_parents(rng, int(n)) for n in rng.integers(1, 10, 3)]
    x = rand_inputs(rng, parents, H=2, dk=6, dv=5)
    x["beta"][:] = 0.0
    x["g"][:] = 0.0
    o, U, G = verify_of(impl, x)
    for r in range(len(parents)):
        for t in range(x["cu"][r], x["cu"][r + 1]):
            for h in range(2):
                S0 = x["ST0"][r, h].T
                np.testing.assert_allclose(o[t, h], S0 @ x["q"][t, h], atol=1e-12)
    np.testing.assert_allclose(U, 0.0, atol=0)
    np.testing.assert_allclose(commit_of(impl, x), x["ST0"], atol=1e-12)


def pin_pure_decay(impl, seed=2):
    """beta = 0: S_t = (prod of a over the root-to-node path) S_0."""
    rng = np.random.default_rng(seed)
    parents = [random_parents(rng, int(n), depth=6) for n in rng.integers(2, 12, 3)]
    x = rand_inputs(rng, parents, H=2, dk=5, dv=7)
    x["beta"][:] = 0.0
    o, U, G = verify_of(impl, x)
    for r, par in enumerate(parents):
        t0 = x["cu"][r]
        for t in range(len(par)):
            anc = ancestors_plus(par, t)
            for h in range(2):
                Gt = sum(x["g"][t0 + j, h] for j in anc)
                np.testing.assert_allclose(G[t0 + t, h], Gt, atol=1e-12)
                want = math.exp(Gt) * (x["ST0"][r, h].T @ x["q"][t0 + t, h])
                np.testing.assert_allclose(o[t0 + t, h], want, atol=1e-12)
    ST = commit_of(impl, x)
    for r in range(len(parents)):
        L = x["plen"][r]
        for h in range(2):
            Gl = sum(x["g"][x["cu"][r] + j, h] for j in x["path"][r, :L])
            np.testing.assert_allclose(ST[r, h], math.exp(Gl) * x["ST0"][r, h], atol=1e-12)


def pin_erasure(impl, seed=3):
    """beta = 1, |k| = 1, q = k: the node's own write is read back exactly, o_t = v_t."""
    rng = np.random.default_rng(seed)
    parents = [random_parents(rng, int(n)) for n in rng.integers(1, 12, 3)]
    x = rand_inputs(rng, parents, H=2, dk=8, dv=6)
    x["beta"][:] = 1.0
    x["q"] = x["k"].copy()
    o, U, G = verify_of(impl, x)
    np.testing.assert_allclose(o, x["v"], atol=1e-12)


def pin_single_node_zero_state(impl, seed=4):
    rng = np.random.default_rng(seed)
    x = rand_inputs(rng, [np.array([-1], np.int32)] * 2, H=3, dk=7, dv=4)
    x["ST0"][:] = 0.0
    o, U, G = verify_of(impl, x)
    for t in range(2):
        for h in range(3):
            b = x["beta"][t, h]
            np.testing.assert_allclose(o[t, h], b * (x["k"][t, h] @ x["q"][t, h]) * x["v"][t, h], atol=1e-13)
            np.testing.assert_allclose(U[t, h], b * x["v"][t, h], atol=1e-13)


def pin_orthonormal_keys(impl, seed=5):
    """Orthonormal keys: earlier writes never interfere with later reads, so with
    gamma_t = exp(G_t):
        u_t = b_t (v_t - gamma_t S_0 k_t)
        o_t = gamma_t S_0 q_t + sum_{j on root..t} (gamma_t / gamma_j) (k_j . q_t) u_j
        S_l = gamma_l S_0 + sum_{j on accepted path} (gamma_l / gamma_j) u_j k_j^T
    """
    rng = np.random.default_rng(seed)
    dk, dv, H = 12, 5, 2
    parents = [random_parents(rng, int(n), depth=7) for n in rng.integers(3, 12, 3)]
    x = rand_inputs(rng, parents, H=H, dk=dk, dv=dv)
    for r, par in enumerate(parents):
        t0 = x["cu"][r]
        for h in range(H):
            Qm, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
            x["k"][t0:t0 + len(par), h] = Qm[:len(par)]
    o, U, G = verify_of(impl, x)
    ST = commit_of(impl, x)
    for r, par in enumerate(parents):
        t0 = x["cu"][r]
        for h in range(H):
            S0 = x["ST0"][r, h].T
            gam = {}
            u = {}
            for t in range(len(par)):
                anc = ancestors_plus(par, t)
                gam[t] = math.exp(sum(x["g"][t0 + j, h] for j in anc))
                u[t] = x["beta"][t0 + t, h] * (x["v"][t0 + t, h] - gam[t] * S0 @ x["k"][t0 + t, h])
            for t in range(len(par)):
                anc = ancestors_plus(par, t)
                qt = x["q"][t0 + t, h]
                want = gam[t] * S0 @ qt
                for j in anc:
                    want = want + (gam[t] / gam[j]) * (x["k"][t0 + j, h] @ qt) * u[j]
                np.testing.assert_allclose(U[t0 + t, h], u[t], atol=1e-12)
                np.testing.assert_allclose(o[t0 + t, h], want, atol=1e-12)
            L = x["plen"][r]
            if L:
                pth = list(x["path"][r, :L])
                l = pth[-1]
                Sl = gam[l] * S0
                for j in pth:
                    Sl = Sl + (gam[l] / gam[j]) * np.outer(u[j], x["k"][t0 + j, h])
            else:
                Sl = S0
            np.testing.assert_allclose(ST[r, h], Sl.T, atol=1e-12)


def pin_linearity(impl, seed=6):
    """For fixed keys, queries, beta and gates the rule is linear in (S_0, v) jointly."""
    rng = np.random.default_rng(seed)
    parents = [random_parents(rng, int(n)) for n in rng.integers(1, 10, 2)]
    x = rand_inputs(rng, parents, H=2, dk=6, dv=6)
    y = dict(x)
    y["ST0"] = rng.normal(size=x["ST0"].shape)
    y["v"] = rng.normal(size=x["v"].shape)
    z = dict(x)
    alpha = 1.7
    z["ST0"] = alpha * x["ST0"] + y["ST0"]
    z["v"] = alpha * x["v"] + y["v"]
    ox, Ux, _ = verify_of(impl, x)
    oy, Uy, _ = verify_of(impl, y)
    oz, Uz, _ = verify_of(impl, z)
    np.testing.assert_allclose(oz, alpha * ox + oy, atol=1e-11)
    np.testing.assert_allclose(Uz, alpha * Ux + Uy, atol=1e-11)
    np.testing.assert_allclose(commit_of(impl, z), alpha * commit_of(impl, x) + commit_of(impl, y), atol=1e-11)


def _literal_step(S, a, b, k, v):
    """The rule in its literal matrix form, S a (I - b k k^T) + b v k^T."""
    d = len(k)
    return a * S @ (np.eye(d) - b * np.outer(k, k)) + b * np.outer(v, k)


def pin_chain_is_sequential_decode(impl, seed=7):
    """A chain verified as a tree equals decoding its tokens one at a time (S carried)."""
    rng = np.random.default_rng(seed)
    n, H, d = 9, 2, 6
    x = rand_inputs(rng, [W.chain_parents(n)], H=H, dk=d, dv=d, paths=[list(range(n))])
    o, U, G = verify_of(impl, x)
    ST = commit_of(impl, x)
    for h in range(H):
        S = x["ST0"][0, h].T.copy()
        for t in range(n):
            S = _literal_step(S, math.exp(x["g"][t, h]), x["beta"][t, h], x["k"][t, h], x["v"][t, h])
            np.testing.assert_allclose(o[t, h], S @ x["q"][t, h], atol=1e-12)
        np.testing.assert_allclose(ST[0, h], S.T, atol=1e-12)


def pin_storeall_bruteforce(impl, seed=8):
    """Store-all: step each node from its parent's stored state (brute force on tiny trees)."""
    rng = np.random.default_rng(seed)
    parents = [random_parents(rng, int(n), depth=6) for n in rng.integers(1, 12, 3)]
    x = rand_inputs(rng, parents, H=2, dk=5, dv=4)
    o, U, G = verify_of(impl, x)
    for r, par in enumerate(parents):
        t0 = x["cu"][r]
        for h in range(2):
            snaps = {}
            for t in range(len(par)):
                Sp = x["ST0"][r, h].T if par[t] < 0 else snaps[int(par[t])]
                a = math.exp(x["g"][t0 + t, h])
                b = x["beta"][t0 + t, h]
                snaps[t] = _literal_step(Sp, a, b, x["k"][t0 + t, h], x["v"][t0 + t, h])
                np.testing.assert_allclose(o[t0 + t, h], snaps[t] @ x["q"][t0 + t, h], atol=1e-12)
                # pseudo-value is the rank-1 part: S_t - a S_parent = u_t k_t^T
                np.testing.assert_allclose(np.outer(U[t0 + t, h], x["k"][t0 + t, h]),
                                           snaps[t] - a * Sp, atol=1e-12)


ALL_PINS = [pin_worked_example, pin_no_write, pin_pure_decay, pin_erasure, pin_single_node_zero_state,
            pin_orthonormal_keys, pin_linearity, pin_chain_is_sequential_decode, pin_storeall_bruteforce]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(impl, pin):
    pin(impl)


# ---------------------------------------------------------------------------
# structural invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("impl", IMPLS)
def test_branch_extraction(impl):
    """A node's output, pseudo-value and log-gate only depend on its root-to-node path."""
    rng = np.random.default_rng(11)
    par = random_parents(rng, 11, depth=5)
    x = rand_inputs(rng, [par], H=2, dk=6, dv=5)
    o, U, G = verify_of(impl, x)
    for t in range(len(par)):
        anc = ancestors_plus(par, t)
        sub = dict(x)
        sub["parent"] = W.chain_parents(len(anc))
        sub["cu"] = np.array([0, len(anc)], np.int32)
        for key in ("q", "k", "v", "beta", "g"):
            sub[key] = x[key][anc]
        so, sU, sG = verify_of(impl, sub)
        np.testing.assert_allclose(so[-1], o[t], atol=1e-12)
        np.testing.assert_allclose(sU[-1], U[t], atol=1e-12)
        np.testing.assert_allclose(sG[-1], G[t], atol=1e-12)


@pytest.mark.parametrize("impl", IMPLS)
def test_topological_relabel(impl):
    rng = np.random.default_rng(12)
    par = W.random_tree_parents(rng, 12, fanout_max=3, depth_max=4)
    x = rand_inputs(rng, [par], H=2, dk=5, dv=5)
    o, U, G = verify_of(impl, x)
    npar, perm = W.random_topological_relabel(rng, par)
    y = dict(x)
    y["parent"] = npar
    for key in ("q", "k", "v", "beta", "g"):
        y[key] = x[key][perm]
    o2, U2, G2 = verify_of(impl, y)
    np.testing.assert_allclose(o2, o[perm], atol=1e-12)
    np.testing.assert_allclose(U2, U[perm], atol=1e-12)
    np.testing.assert_allclose(G2, G[perm], atol=1e-12)


@pytest.mark.parametrize("impl", IMPLS)
def test_commit_state_reproduces_accepted_output(impl):
    """Rebuilt state of a path ending at l, applied to q_l, equals verify's o_l."""
    rng = np.random.default_rng(13)
    parents = [random_parents(rng, int(n)) for n in rng.integers(2, 12, 4)]
    x = rand_inputs(rng, parents, H=2, dk=6, dv=6)
    o, _, _ = verify_of(impl, x)
    ST = commit_of(impl, x)
    for r in range(len(parents)):
        L = x["plen"][r]
        if L == 0:
            continue
        l = x["cu"][r] + x["path"][r, L - 1]
        for h in range(2):
            np.testing.assert_allclose(ST[r, h].T @ x["q"][l, h], o[l, h], atol=1e-12)


def wy_fp64(x):
    """Tree-structured WY form, fp64, test-only: one unit-lower-triangular system per
    (request, head) for the pseudo-values, outputs from S_0 q plus masked pseudo-value terms.
        (I + A) U = R,   A[t,j] = b_t e^{G_t - G_j} (k_t . k_j)  for j a strict ancestor of t
        R_t = b_t (v_t - e^{G_t} S_0 k_t)
        o_t = e^{G_t} S_0 q_t + sum_{j ancestor-or-self} e^{G_t - G_j} (q_t . k_j) u_j
    """
    B, H = x["ST0"].shape[:2]
    T = int(x["cu"][-1])
    dv = x["v"].shape[-1]
    o = np.zeros((T, H, dv))
    U = np.zeros((T, H, dv))
    for r in range(B):
        t0, t1 = int(x["cu"][r]), int(x["cu"][r + 1])
        n = t1 - t0
        if n == 0:
            continue
        par = x["parent"][t0:t1]
        ancm = np.zeros((n, n), bool)
        for t in range(n):
            for j in ancestors_plus(par, t):
                ancm[t, j] = True
        strict = ancm & ~np.eye(n, dtype=bool)
        for h in range(H):
            S0 = x["ST0"][r, h].T
            K = x["k"][t0:t1, h]
            Q = x["q"][t0:t1, h]
            V = x["v"][t0:t1, h]
            b = x["beta"][t0:t1, h]
            Gt = np.array([sum(x["g"][t0 + j, h] for j in ancestors_plus(par, t)) for t in range(n)])
            D = np.exp(Gt[:, None] - Gt[None, :])
            A = np.where(strict, b[:, None] * D * (K @ K.T), 0.0)
            P = np.where(ancm, D * (Q @ K.T), 0.0)
            R = b[:, None] * (V - np.exp(Gt)[:, None] * (K @ S0.T))
            Uw = np.linalg.solve(np.eye(n) + A, R)
            o[t0:t1, h] = np.exp(Gt)[:, None] * (Q @ S0.T) + P @ Uw
            U[t0:t1, h] = Uw
    return o, U


def test_wy_identity_matches_replay():
    """The derivation the CUDA path implements agrees with the replay in fp64."""
    rng = np.random.default_rng(14)
    parents = [random_parents(rng, int(n), depth=6) for n in rng.integers(1, 20, 5)]
    x = rand_inputs(rng, parents, H=3, dk=9, dv=7)
    o, U, _ = verify_of("c", x)
    ow, Uw = wy_fp64(x)
    np.testing.assert_allclose(ow, o, atol=1e-11)
    np.testing.assert_allclose(Uw, U, atol=1e-11)


def test_c_matches_numpy_ragged_with_empty_requests():
    tb = W.make_random_batch(seed=15, B=7, H=2, d=8, n_range=(1, 12), empty_every=3)
    inp = oracle.batch_inputs(tb)
    oc, Uc, Gc = oracle.verify(**inp)
    on, Un, Gn = replay.verify(inp["ST0"], inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"],
                               inp["parent"], inp["cu_nodes"])
    np.testing.assert_allclose(oc, on, atol=1e-12)
    np.testing.assert_allclose(Uc, Un, atol=1e-12)
    np.testing.assert_allclose(Gc, Gn, atol=1e-12)
    Sc = oracle.commit(inp["ST0"], inp["k"], inp["v"], inp["beta"], inp["g"], tb.parent, tb.cu_nodes,
                       tb.path, tb.path_len)
    Sn = replay.commit(inp["ST0"], inp["k"], inp["v"], inp["beta"], inp["g"], tb.parent, tb.cu_nodes,
                       tb.path, tb.path_len)
    np.testing.assert_allclose(Sc, Sn, atol=1e-12)


def test_sampled_pairs_match_full():
    tb = W.make_random_batch(seed=16, B=5, H=3, d=8, n_range=(1, 10))
    inp = oracle.batch_inputs(tb)
    of, Uf, Gf = oracle.verify(**inp)
    pairs = [14, 2, 7]
    oc, Uc, Gc = oracle.verify(**inp, pairs=pairs)
    row = 0
    for p in pairs:
        r, h = divmod(p, 3)
        t0, t1 = tb.cu_nodes[r], tb.cu_nodes[r + 1]
        np.testing.assert_array_equal(oc[row:row + t1 - t0], of[t0:t1, h])
        np.testing.assert_array_equal(Uc[row:row + t1 - t0], Uf[t0:t1, h])
        np.testing.assert_array_equal(Gc[row:row + t1 - t0], Gf[t0:t1, h])
        row += t1 - t0
    Sf = oracle.commit(inp["ST0"], inp["k"], inp["v"], inp["beta"], inp["g"], tb.parent, tb.cu_nodes,
                       tb.path, tb.path_len)
    Sc = oracle.commit(inp["ST0"], inp["k"], inp["v"], inp["beta"], inp["g"], tb.parent, tb.cu_nodes,
                       tb.path, tb.path_len, pairs=pairs)
    for i, p in enumerate(pairs):
        np.testing.assert_array_equal(Sc[i], Sf[p // 3, p % 3])


@pytest.mark.parametrize("impl", IMPLS)
def test_invalid_tree_and_path_rejected(impl):
    rng = np.random.default_rng(17)
    x = rand_inputs(rng, [W.chain_parents(4)], H=1, dk=4, dv=4, paths=[[0, 1]])
    bad = dict(x)
    bad["parent"] = np.array([-1, 0, 2, 1], np.int32)  # node 2 names itself as parent
    with pytest.raises(ValueError):
        verify_of(impl, bad)
    bad["parent"] = np.array([0, 0, 1, 2], np.int32)  # root names node 0
    with pytest.raises(ValueError):
        verify_of(impl, bad)
    for pth in ([1, 2], [0, 2], [0, 4], [-1, 0]):
        y = dict(x)
        y["path"] = np.array([pth], np.int32)
        y["plen"] = np.array([2], np.int32)
        with pytest.raises(ValueError):
            commit_of(impl, y)


# ---------------------------------------------------------------------------
# the pins catch planted mistakes (planted in the NumPy twin only, on the CPU)
# ---------------------------------------------------------------------------

def _mut_drop_write(S, a, b, k, v):
    Sk = S @ k
    return a * S - a * b * np.outer(Sk, k), b * (v - a * Sk)


def _mut_erase_sign(S, a, b, k, v):
    Sk = S @ k
    return a * S + a * b * np.outer(Sk, k) + b * np.outer(v, k), b * (v - a * Sk)


def _mut_transposed_state(S, a, b, k, v):
    Sk = S.T @ k
    return a * S - a * b * np.outer(Sk, k) + b * np.outer(v, k), b * (v - a * Sk)


def _mut_gate_missing_on_erase(S, a, b, k, v):
    Sk = S @ k
    return a * S - b * np.outer(Sk, k) + b * np.outer(v, k), b * (v - Sk)


def _mut_beta_missing_in_u(S, a, b, k, v):
    Sk = S @ k
    return a * S - a * b * np.outer(Sk, k) + b * np.outer(v, k), v - a * Sk


def _mut_gate_squared(S, a, b, k, v):
    Sk = S @ k
    return a * a * S - a * b * np.outer(Sk, k) + b * np.outer(v, k), b * (v - a * Sk)


def _mut_chain_instead_of_tree(parent_r, t):
    return list(range(t + 1))


def _mut_skip_root(parent_r, t):
    out = []
    x = t
    while x >= 0:
        out.append(x)
        x = int(parent_r[x])
    return out[::-1][1:] if len(out) > 1 else out


@pytest.mark.parametrize("mutation", [
    ("rule_step", _mut_drop_write), ("rule_step", _mut_erase_sign), ("rule_step", _mut_transposed_state),
    ("rule_step", _mut_gate_missing_on_erase), ("rule_step", _mut_beta_missing_in_u),
    ("rule_step", _mut_gate_squared), ("_root_path", _mut_chain_instead_of_tree),
    ("_root_path", _mut_skip_root)], ids=lambda m: m[1].__name__)
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    name, fn = mutation
    monkeypatch.setattr(replay, name, fn)
    failures = 0
    for pin in ALL_PINS:
        try:
            pin("numpy")
        except (AssertionError, ValueError):  # a shape error is also a caught mistake
            failures += 1
    assert failures >= 1, f"no pin caught the planted mistake {fn.__name__}"
