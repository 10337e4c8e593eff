"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and compare it with
the CPU oracle on the same seeded inputs.

Tolerances (stated for fp32 state / fp32 accumulation with bf16 q, k, v):
  outputs o and pseudo-values U : max |x - x_ref| <= 2e-3 * (max |x_ref| + 1)
  committed state               : ||ST - ST_ref||_F / ||ST_ref||_F <= 1e-3
  cumulative log-gate G         : |G - G_ref| <= 1e-5 * (|G_ref| + 1)   (fp32 sum of <= 64 terms)
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_deltanet_tree_03_b300 import binding as gb
from gated_deltanet_tree_03_b300 import device as gd

O_TOL = 2e-3
S_TOL = 1e-3
G_TOL = 1e-5

VERIFY_FNS = {"wy": gb.gdn_tree_verify, "simt": gb.gdn_tree_verify_simt}


def run_gpu(tb, verify: str = "wy", commit: bool = True, fill=float("nan"), max_nodes=None, max_path=None):
    """Run verify (and commit) on cuda:0 for a host TreeBatch. Returns numpy results."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = gd.upload(tb)
    out = gd.alloc_outputs(tb, fill=fill)
    mn = tb.max_nodes if max_nodes is None else max_nodes
    mp = tb.max_path if max_path is None else max_path
    args = (d["ST"], d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"], d["cu_nodes"],
            tb.B, tb.H, tb.T, tb.dk, tb.dv, mn)
    snap = None
    if verify == "storeall":
        snap = torch.full((max(tb.T, 1), tb.H, tb.dk, tb.dv), float("nan"), device="cuda")
        gb.gdn_tree_verify_storeall(*args, snap, out["o"], out["U"], out["G"], out["status"])
    else:
        VERIFY_FNS[verify](*args, out["o"], out["U"], out["G"], out["status"])
    if commit:
        if verify == "storeall":
            gb.gdn_tree_commit_storeall(d["ST"], snap, d["parent"], d["cu_nodes"], d["path"], d["path_len"],
                                        tb.B, tb.H, tb.T, tb.dk, tb.dv, mp, out["status"])
        else:
            gb.gdn_tree_commit(d["ST"], out["U"], out["G"], d["k"], d["parent"], d["cu_nodes"], d["path"],
                               d["path_len"], tb.B, tb.H, tb.T, tb.dk, tb.dv, mp, out["status"])
    torch.cuda.synchronize()
    res = {"o": out["o"][:tb.T].cpu().numpy(), "U": out["U"][:tb.T].cpu().numpy(),
           "G": out["G"][:tb.T].cpu().numpy(), "ST": d["ST"].cpu().numpy(),
           "status": int(out["status"][0].item())}
    if snap is not None:
        res["snap"] = snap[:tb.T].cpu().numpy()
    return res


def sample_pairs(tb, n: int, seed: int = 0) -> list[int]:
    total = tb.B * tb.H
    if total <= n:
        return list(range(total))
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(total, size=n - 2, replace=False).tolist())
    pick.update([0, total - 1])
    return sorted(pick)


def gather_rows(tb, arr, pairs):
    """Rows of a [T,H,...] array for the listed pairs, in the oracle's compact order."""
    rows = []
    for p in pairs:
        r, h = divmod(p, tb.H)
        rows.append(arr[tb.cu_nodes[r]:tb.cu_nodes[r + 1], h])
    return np.concatenate(rows, axis=0) if rows else arr[:0, 0]


def max_err(x, ref):
    if ref.size == 0:
        return 0.0, 1.0
    return float(np.max(np.abs(x.astype(np.float64) - ref))), float(np.max(np.abs(ref)))


def check_verify(tb, res, pairs=None, tag=""):
    inp = oracle.batch_inputs(tb)
    if pairs is None:
        o_ref, U_ref, G_ref = oracle.verify(**inp)
        o, U, G = res["o"], res["U"], res["G"]
    else:
        o_ref, U_ref, G_ref = oracle.verify(**inp, pairs=pairs)
        o, U, G = (gather_rows(tb, res[key], pairs) for key in ("o", "U", "G"))
    for name, x, ref in (("o", o, o_ref), ("U", U, U_ref)):
        assert np.all(np.isfinite(x)), f"{tag}: non-finite {name}"
        e, m = max_err(x, ref)
        assert e <= O_TOL * (m + 1.0), f"{tag}: {name} max err {e:.3e} > {O_TOL}*({m:.3f}+1)"
    gerr = np.abs(G.astype(np.float64) - G_ref)
    assert np.all(gerr <= G_TOL * (np.abs(G_ref) + 1)), f"{tag}: G err {gerr.max():.3e}"
    return max_err(o, o_ref)


def check_commit(tb, res, pairs=None, tag=""):
    inp = oracle.batch_inputs(tb)
    args = (inp["ST0"], inp["k"], inp["v"], inp["beta"], inp["g"], tb.parent, tb.cu_nodes, tb.path,
            tb.path_len)
    if pairs is None:
        ref = oracle.commit(*args)
        got = res["ST"].astype(np.float64)
    else:
        ref = oracle.commit(*args, pairs=pairs)
        flat = res["ST"].reshape(tb.B * tb.H, tb.dk, tb.dv)
        got = flat[np.asarray(pairs)].astype(np.float64)
    assert np.all(np.isfinite(got)), f"{tag}: non-finite state"
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    assert rel <= S_TOL, f"{tag}: committed state rel Frobenius err {rel:.3e} > {S_TOL}"
    return rel
