"""Pins for the serving-layout oracle (``oracle.serving``): state-pool slots, grouped q/k heads,
the query scale and the gate pre-activations.

* the gate maps against closed forms and identities of softplus and sigmoid that a slip (a
  wrong sign, a missing exp, the wrong branch of the stable form) breaks: softplus(0) = ln 2,
  softplus(x) - softplus(-x) = x, softplus' = sigmoid, sigmoid(x) + sigmoid(-x) = 1, and
  exp(g) = (1 + e^x)^(-e^A_log) for the decay the gate forms;
* the whole serving verify / commit against a brute-force token-by-token replay with the
  slot and head mapping written out per (request, head), through the NumPy twin's single rule
  step rather than the C oracle;
* invariants: permuting the pool together with the slots changes nothing, the output is
  linear in the query scale while U and G do not move, the plain layout is the special case
  (identity slots, H_qk = H, scale 1), and padding requests produce nothing and commit nothing.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import replay, serving
from gated_deltanet_tree_03_b300 import workloads as W


# ---------------------------------------------------------------------------
# gate maps
# ---------------------------------------------------------------------------

def test_softplus_closed_forms_and_identities():
    assert serving.softplus(0.0) == pytest.approx(math.log(2.0), abs=1e-16)
    x = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(serving.softplus(x) - serving.softplus(-x), x, atol=1e-13)
    # large arguments: no overflow, ln(1 + e^x) -> x
    assert serving.softplus(800.0) == 800.0
    assert 0.0 <= serving.softplus(-800.0) < 1e-300
    # the derivative of softplus is the logistic sigmoid (central differences)
    h = 1e-5
    fd = (serving.softplus(x + h) - serving.softplus(x - h)) / (2 * h)
    np.testing.assert_allclose(fd, serving.sigmoid(x), atol=1e-9)


def test_sigmoid_closed_forms_and_symmetry():
    assert serving.sigmoid(0.0) == 0.5
    x = np.linspace(-40, 40, 801)
    np.testing.assert_allclose(serving.sigmoid(x) + serving.sigmoid(-x), 1.0, atol=1e-15)
    with np.errstate(over="raise"):
        assert serving.sigmoid(-800.0) == 0.0
        assert serving.sigmoid(800.0) == 1.0
    np.testing.assert_allclose(serving.sigmoid(np.log(3.0)), 0.75, atol=1e-15)  # 1/(1 + 1/3)


@pytest.mark.parametrize("c", [1.0, 2.0, 3.0, 7.5])
def test_gate_decay_is_a_power_of_the_logistic(c):
    """a = exp(g) = exp(-c ln(1 + e^x)) = (1 + e^x)^-c, x = a_raw + dt_bias, c = e^A_log."""
    rng = np.random.default_rng(3)
    a_raw = rng.normal(size=(9, 3))
    dt_bias = np.array([-4.0, 0.0, 1.5])
    b_raw = rng.normal(size=(9, 3)) * 3
    g, beta = serving.gate_beta(a_raw, b_raw, np.full(3, math.log(c)), dt_bias)
    x = a_raw + dt_bias[None, :]
    np.testing.assert_allclose(np.exp(g), (1.0 + np.exp(x)) ** -c, rtol=1e-12)
    assert np.all(g <= 0)
    np.testing.assert_allclose(beta, 1.0 / (1.0 + np.exp(-b_raw)), rtol=1e-14)


# ---------------------------------------------------------------------------
# serving verify / commit
# ---------------------------------------------------------------------------

def _brute_serving(tb, sv, gates: bool):
    """Token-by-token replay of every node's root-to-node path with the layout written out:
    state pool[slot[r], h] (stored transposed), q/k head h // (H / H_qk), scaled query."""
    H, grp = tb.H, tb.H // sv.H_qk
    q, k, v = W.bf16_bits_to_f32(sv.q).astype(float), W.bf16_bits_to_f32(sv.k).astype(float), tb.v_f32().astype(float)
    if gates:
        x = sv.a_raw.astype(float) + sv.dt_bias.astype(float)[None, :]
        a = (1.0 + np.exp(x)) ** (-np.exp(sv.A_log.astype(float)))[None, :]
        beta = 1.0 / (1.0 + np.exp(-sv.b_raw.astype(float)))
    else:
        a, beta = np.exp(tb.g.astype(float)), tb.beta.astype(float)
    o = np.full((tb.T, H, tb.dv), np.nan)
    for r in range(tb.B):
        if sv.slot[r] < 0:
            continue
        t0 = int(tb.cu_nodes[r])
        par = tb.request_parent(r)
        for h in range(H):
            for t in range(tb.n_nodes(r)):
                S = sv.pool[sv.slot[r], h].astype(float).T
                chain = []
                x_ = t
                while x_ >= 0:
                    chain.append(x_)
                    x_ = int(par[x_])
                for j in reversed(chain):
                    S, _ = replay.rule_step(S, a[t0 + j, h], beta[t0 + j, h], k[t0 + j, h // grp], v[t0 + j, h])
                o[t0 + t, h] = S @ (sv.q_scale * q[t0 + t, h // grp])
    return o


def _serving_args(tb, sv):
    return (sv.pool, sv.slot, W.bf16_bits_to_f32(sv.q), W.bf16_bits_to_f32(sv.k), tb.v_f32(), tb.beta, tb.g,
            tb.parent, tb.cu_nodes)


@pytest.mark.parametrize("H,H_qk,gates", [(4, 2, True), (4, 1, False), (6, 3, True), (2, 2, False)])
def test_serving_verify_matches_brute_force_replay(H, H_qk, gates):
    tb, sv = W.make_serving_batch(seed=11 + H + H_qk, B=5, H=H, H_qk=H_qk, d=8, n_range=(1, 7), pad_every=4)
    o, U, G = serving.verify(*_serving_args(tb, sv), q_scale=sv.q_scale, gates=sv.gates if gates else None)
    ref = _brute_serving(tb, sv, gates)
    live_rows = np.isfinite(ref[:, 0, 0])
    assert live_rows.any() and not live_rows.all()  # both live and padding requests present
    np.testing.assert_allclose(o[live_rows], ref[live_rows], atol=1e-12)
    assert np.all(np.isnan(o[~live_rows])) and np.all(np.isnan(U[~live_rows])) and np.all(np.isnan(G[~live_rows]))


def test_serving_commit_matches_brute_force_and_leaves_other_slots():
    tb, sv = W.make_serving_batch(seed=5, B=6, H=4, H_qk=2, d=8, n_range=(2, 8), pad_every=3)
    new = serving.commit(sv.pool, sv.slot, W.bf16_bits_to_f32(sv.k), tb.v_f32(), tb.beta, tb.g, tb.parent,
                         tb.cu_nodes, tb.path, tb.path_len, gates=sv.gates)
    x = sv.a_raw.astype(float) + sv.dt_bias.astype(float)[None, :]
    a = (1.0 + np.exp(x)) ** (-np.exp(sv.A_log.astype(float)))[None, :]
    beta = 1.0 / (1.0 + np.exp(-sv.b_raw.astype(float)))
    k, v = W.bf16_bits_to_f32(sv.k).astype(float), tb.v_f32().astype(float)
    touched = set()
    for r in range(tb.B):
        s = int(sv.slot[r])
        if s < 0:
            continue
        touched.add(s)
        t0 = int(tb.cu_nodes[r])
        for h in range(tb.H):
            S = sv.pool[s, h].astype(float).T
            for i in range(int(tb.path_len[r])):
                j = t0 + int(tb.path[r, i])
                S, _ = replay.rule_step(S, a[j, h], beta[j, h], k[j, h // 2], v[j, h])
            np.testing.assert_allclose(new[s, h], S.T, atol=1e-12)
    for s in range(sv.pool.shape[0]):
        if s not in touched:
            assert np.array_equal(new[s], sv.pool[s].astype(float))


def test_pool_permutation_invariance_and_plain_special_case():
    tb, sv = W.make_serving_batch(seed=8, B=4, H=2, H_qk=2, d=8, n_range=(1, 6))
    args = list(_serving_args(tb, sv))
    o, U, G = serving.verify(*args)
    perm = np.random.default_rng(0).permutation(sv.pool.shape[0])
    inv = np.argsort(perm)
    args_p = list(args)
    args_p[0] = sv.pool[perm]          # pool_p[i] = pool[perm[i]]
    args_p[1] = inv[sv.slot].astype(np.int32)  # so pool_p[slot_p[r]] = pool[slot[r]]
    o2, U2, G2 = serving.verify(*args_p)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(U, U2)
    # plain layout: states in request order, equal head counts, no scale, given gates
    inp = oracle.batch_inputs(tb)
    inp.update(ST0=sv.pool[sv.slot].astype(float), q=args[2].astype(float), k=args[3].astype(float))
    o3, U3, G3 = oracle.verify(**inp)
    np.testing.assert_array_equal(o, o3)
    np.testing.assert_array_equal(G, G3)


def test_output_is_linear_in_the_query_scale():
    tb, sv = W.make_serving_batch(seed=9, B=3, H=4, H_qk=4, d=8, n_range=(1, 6))
    args = _serving_args(tb, sv)
    o1, U1, G1 = serving.verify(*args, q_scale=1.0)
    o2, U2, G2 = serving.verify(*args, q_scale=0.3125)
    np.testing.assert_allclose(o2, 0.3125 * o1, atol=1e-14)
    np.testing.assert_array_equal(U1, U2)
    np.testing.assert_array_equal(G1, G2)
