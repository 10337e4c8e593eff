#!/usr/bin/env python3
"""Benchmark: draft-node verifications/s for GDN tree verify + commit on B300.

One step = one pass of the whole hot path over one layer's batch: gdn_tree_verify (all
nodes, all heads) followed by gdn_tree_commit (accepted paths), both through the C ABI.

Default workload: the depth-3 chain setting (bonus + 3 drafts = 4 nodes per request),
256 requests, 32 heads, d_k = d_v = 128, fp32 state, bf16 q/k/v; several layers' input sets
are resident and rotated so every step streams its state from HBM (each layer's state is
512 MiB, larger than the 126 MB L2).

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU fp64 replay oracle instead
(a deliberately slow baseline), on the same workload, metric and unit.

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no data-path
collective): the step time is the max over ranks and ``value`` counts all ranks' nodes.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft-node verifications/sec (verify+commit) and achieved HBM GB/s vs B300 peak"
UNIT = "node-verifications/s"
KERNEL_SOURCES = {
    "verify": ["verify_stream.cuh", "verify_tc.cuh", "verify_simt.cuh", "common.cuh", "ptx.cuh", "bounds.cuh"],
    "commit": ["commit.cuh", "common.cuh", "ptx.cuh", "bounds.cuh"],
}
NOMINAL_HBM_GBS = 8000.0  # the B300 HBM3e figure the roofline target is quoted against


# ---------------------------------------------------------------------------
# algorithmic byte / flop model (per launch)
# ---------------------------------------------------------------------------

def verify_bytes(tb) -> int:
    """State read once + per (node, head): q, k, v in; beta, g in; o, U out; G out."""
    per_node_head = 2 * tb.dk * 2 + tb.dv * 2 + 8 + 2 * tb.dv * 4 + 4
    return tb.B * tb.H * tb.dk * tb.dv * 4 + tb.T * tb.H * per_node_head + tb.T * 4 + (tb.B + 1) * 4


def commit_bytes(tb) -> int:
    """State read + written once per (request, head) with a non-empty path, plus the path's
    u (fp32), k (bf16) and G."""
    L = tb.path_len.astype(np.int64)
    active = int(np.sum(L > 0))
    return active * tb.H * 2 * tb.dk * tb.dv * 4 + int(L.sum()) * tb.H * (tb.dv * 4 + tb.dk * 2 + 4)


def fused_bytes(tb) -> int:
    """gdn_tree_commit_verify with the same tree on both sides of the step: the verify's and the
    commit's bytes, less the one state read the fusion removes per committed (request, head)."""
    active = int(np.sum(tb.path_len.astype(np.int64) > 0))
    return verify_bytes(tb) + commit_bytes(tb) - active * tb.H * tb.dk * tb.dv * 4


def attention_bytes(ab) -> int:
    """Tree-bias attention: every prefix key and value read once per (request, key/value head),
    the draft nodes' q, k, v read once, o (fp32) written once."""
    return (2 * ab.P * ab.Hkv * ab.d * 2 + ab.T * ab.Hq * ab.d * 2 + 2 * ab.T * ab.Hkv * ab.d * 2
            + ab.T * ab.Hq * ab.d * 4 + ab.T * 4 + 2 * (ab.B + 1) * 4)


def attention_flops(ab) -> int:
    """Useful multiply-adds x 2 of Q.K^T and P.V: per query row, (prefix + root-path) keys."""
    depth = np.zeros(ab.T, np.int64)
    for r in range(ab.B):
        t0 = int(ab.cu_nodes[r])
        for t in range(int(ab.cu_nodes[r + 1]) - t0):
            p = int(ab.parent[t0 + t])
            depth[t0 + t] = 1 if p < 0 else depth[t0 + p] + 1
    plen = np.repeat(np.diff(ab.cu_prefix), np.diff(ab.cu_nodes))
    return int(4 * ab.d * ab.Hq * np.sum(plen + depth))


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1800.0)),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "source": "fallback"}


def kernel_src_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        p = os.path.join(ROOT, "gated_deltanet_tree_03_b300", "csrc", name)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:12]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel source (lines: kernel workload bytes_per_launch src_sha)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_src_sha(kernel)
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload \
                    and parts[3] == sha:
                return float(parts[2])
    return None


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(gpu_index)], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (harness only; the path itself has no collective)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_layers(rank: int, n_layers: int) -> list[int]:
    """Input-set (layer) indices owned by one rank: disjoint across ranks, so ranks process
    independent batches."""
    return [rank * n_layers + i for i in range(n_layers)]


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

WORKLOAD_NAMES = {
    0: ("chain3_d32", "chain of 3 draft nodes, B=1, H=1, d_k=d_v=32"),
    1: ("chain4", "depth-3 chain (4 nodes incl. bonus), B={B}, H=32, d_k=d_v=128, fp32 state, bf16 q/k/v"),
    2: ("rootbranch6", "6-node root-branch tree, B={B}, H=48, d_k=d_v=128, fp32 state, bf16 q/k/v"),
    3: ("ragged16to64", "ragged random trees of 16-64 nodes (fanout<=4, depth<=8), B={B}, H=32, d_k=d_v=128"),
    4: ("tree32", "32-node random trees (fanout<=3, depth<=6), B={B}, H=32, d_k=d_v=128, gate a~U(0.85,1)"),
}


def workload_name(cfg: int, batch: int) -> str:
    return WORKLOAD_NAMES[cfg][1].format(B=batch)


def workload_key(cfg: int, batch: int) -> str:
    """Short label of a workload and batch, as used in profiles/traffic.txt."""
    return f"{WORKLOAD_NAMES[cfg][0]}_B{batch}"


def make_layers(cfg: int, batch: int, layer_ids):
    from gated_deltanet_tree_03_b300 import workloads as W
    return [W.make_config(cfg, batch=batch, layer=l) for l in layer_ids]


def sub_batch(tb, r0: int, r1: int):
    """Requests r0..r1-1 of a TreeBatch (all heads), as a new TreeBatch."""
    from gated_deltanet_tree_03_b300.workloads import TreeBatch
    t0, t1 = int(tb.cu_nodes[r0]), int(tb.cu_nodes[r1])
    return TreeBatch(B=r1 - r0, H=tb.H, dk=tb.dk, dv=tb.dv, parent=tb.parent[t0:t1].copy(),
                     cu_nodes=(tb.cu_nodes[r0:r1 + 1] - t0).astype(np.int32), path=tb.path[r0:r1].copy(),
                     path_len=tb.path_len[r0:r1].copy(), ST0=tb.ST0[r0:r1].copy(), q=tb.q[t0:t1].copy(),
                     k=tb.k[t0:t1].copy(), v=tb.v[t0:t1].copy(), beta=tb.beta[t0:t1].copy(),
                     g=tb.g[t0:t1].copy(), name=tb.name + f"[{r0}:{r1}]")


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_step(sb):
    import oracle
    inp = oracle.batch_inputs(sb)
    oracle.verify(**inp)
    oracle.commit(inp["ST0"], inp["k"], inp["v"], inp["beta"], inp["g"], sb.parent, sb.cu_nodes, sb.path,
                  sb.path_len)


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(tb, target_s: float = 12.0) -> dict:
    """Time the oracle as it stands (OpenMP over pairs, all host cores) on a bounded sample of
    the workload: the first R requests with all heads, R sized for about target_s seconds."""
    import oracle
    one = sub_batch(tb, 0, 1)
    t = time.perf_counter()
    oracle_step(one)
    t1 = max(time.perf_counter() - t, 1e-4)
    R = int(max(1, min(tb.B, target_s / t1)))
    sb = sub_batch(tb, 0, R)
    t = time.perf_counter()
    oracle_step(sb)
    dt = time.perf_counter() - t
    nodes = int(sb.cu_nodes[-1])
    return {"value": nodes / dt, "unit": UNIT, "cores": oracle.max_threads(), "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"first {R} of {tb.B} requests x all {tb.H} heads (verify + commit replay, fp64), "
                      f"{dt:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    tb = make_layers(args.config, args.batch, [0])[0]
    steps, warmup = args.steps, args.warmup
    R = args.ref_requests
    samples = [sub_batch(tb, (i * R) % tb.B, (i * R) % tb.B + R) for i in range(min(tb.B // R, 64))]
    for i in range(warmup):
        oracle_step(samples[i % len(samples)])
    nodes = 0
    t = time.perf_counter()
    for i in range(steps):
        sb = samples[i % len(samples)]
        oracle_step(sb)
        nodes += int(sb.cu_nodes[-1])
    dt = time.perf_counter() - t
    value = nodes / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(args.config, tb.B), "sample_per_step": f"{R} request(s) x {tb.H} heads"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "cpu_model": cpu_model(),
                             "kind": "oracle",
                             "sample": f"{R} request(s) x all {tb.H} heads per step, verify + commit replay"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

# every preset batch, as the line's "workloads" object: (config, batch, layers rotated)
WORKLOAD_SET = [(0, 1, 4), (1, 256, 4), (2, 1, 4), (2, 64, 4), (3, 128, 4), (4, 1, 48), (4, 8, 48), (4, 32, 48),
                (4, 128, 48), (4, 256, 48), (4, 512, 48)]
L2_BYTES = 126 * 2 ** 20
FLUSH_BYTES = 512 * 2 ** 20


def layer_bytes(shape) -> int:
    """HBM bytes one layer's verify + commit touch: state, node block, outputs."""
    return shape.B * shape.H * shape.dk * shape.dv * 4 + shape.T * shape.H * (2 * shape.dk * 2 + shape.dv * 2 + 8 +
                                                                              2 * shape.dv * 4 + 4)


def time_workloads(gb, dev, stream, peaks, reps: int) -> dict:
    """Every preset batch of the synthetic workloads, each over its own rotated layers (own state,
    q, k, v, beta, g per layer; the batch sweep uses its 48 layers). Per pass (one layer's verify
    then commit) the kernels are timed with CUDA events on the launching stream; when the rotated
    working set is under 4x the L2, a 512 MB scratch write before each pass (outside the events)
    evicts the previous passes' data. Values are drawn on the device with the presets' recipe."""
    import torch
    from gated_deltanet_tree_03_b300 import workloads as W
    scratch = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = {}
    for cfg, B, nl in WORKLOAD_SET:
        shapes = [W.config_shape(cfg, B, l) for l in range(nl)]
        layers = [W.draw_values_device(sh, seed=1000 * cfg + l, device=dev) for l, sh in enumerate(shapes)]
        outs = [{"o": torch.empty(sh.T, sh.H, sh.dv, device=dev), "U": torch.empty(sh.T, sh.H, sh.dv, device=dev),
                 "G": torch.empty(sh.T, sh.H, device=dev), "U2": torch.empty(sh.T, sh.H, sh.dv, device=dev),
                 "G2": torch.empty(sh.T, sh.H, device=dev)} for sh in shapes]
        status = torch.zeros(4, dtype=torch.int32, device=dev)
        ws = sum(layer_bytes(sh) for sh in shapes)
        flush = ws < 4 * L2_BYTES

        def verify(j, U="U", G="G"):
            sh, d, o = shapes[j], layers[j], outs[j]
            gb.gdn_tree_verify(d["ST"], d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"], d["cu_nodes"], sh.B,
                               sh.H, sh.T, sh.dk, sh.dv, sh.max_nodes, o["o"], o[U], o[G], status, stream)

        def commit(j, U="U", G="G"):
            sh, d, o = shapes[j], layers[j], outs[j]
            gb.gdn_tree_commit(d["ST"], o[U], o[G], d["k"], d["parent"], d["cu_nodes"], d["path"], d["path_len"],
                               sh.B, sh.H, sh.T, sh.dk, sh.dv, sh.max_path, status, stream)

        for j in range(min(nl, 3)):
            verify(j)
            commit(j)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
        for r in range(reps):
            if flush:
                scratch.fill_(float(r))
            j = r % nl
            ev[r][0].record(stream)
            verify(j)
            ev[r][1].record(stream)
            commit(j)
            ev[r][2].record(stream)
        torch.cuda.synchronize()
        v_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / reps
        c_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / reps
        # commit folded into the next verify (gdn_tree_commit_verify); pseudo-values alternate between
        # two buffers per layer so that each call commits the previous call's accepted paths
        cur = [0] * nl
        for j in range(nl):
            verify(j)

        def fused(j):
            sh, d, o = shapes[j], layers[j], outs[j]
            (Up, Gp), (Un, Gn) = ((o["U"], o["G"]), (o["U2"], o["G2"]))[::1 if cur[j] == 0 else -1]
            gb.gdn_tree_commit_verify(d["ST"], Up, Gp, d["k"], d["parent"], d["cu_nodes"], d["path"], d["path_len"],
                                      sh.T, sh.max_path, d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"],
                                      d["cu_nodes"], sh.B, sh.H, sh.T, sh.dk, sh.dv, sh.max_nodes, o["o"], Un, Gn,
                                      status, stream)
            cur[j] = 1 - cur[j]

        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
        for r in range(reps):
            if flush:
                scratch.fill_(float(r))
            fev[r][0].record(stream)
            fused(r % nl)
            fev[r][1].record(stream)
        torch.cuda.synchronize()
        f_ms = sum(e[0].elapsed_time(e[1]) for e in fev) / reps
        # back-to-back steps (no flush) from Python and replayed from CUDA graphs: how much of a
        # small batch's step is host time
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for r in range(reps):
            verify(r % nl)
            commit(r % nl)
        e1.record(stream)
        torch.cuda.synchronize()
        eager_ms = e0.elapsed_time(e1) / reps
        graph_ms = None
        if B <= 8:
            graphs = []
            for j in range(nl):
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    cs = torch.cuda.current_stream()
                    sh, d, o = shapes[j], layers[j], outs[j]
                    gb.gdn_tree_verify(d["ST"], d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"],
                                       d["cu_nodes"], sh.B, sh.H, sh.T, sh.dk, sh.dv, sh.max_nodes, o["o"], o["U"],
                                       o["G"], status, cs)
                    gb.gdn_tree_commit(d["ST"], o["U"], o["G"], d["k"], d["parent"], d["cu_nodes"], d["path"],
                                       d["path_len"], sh.B, sh.H, sh.T, sh.dk, sh.dv, sh.max_path, status, cs)
                graphs.append(gr)
            for j in range(nl):
                graphs[j].replay()
            torch.cuda.synchronize()
            e0.record()
            for r in range(reps):
                graphs[r % nl].replay()
            e1.record()
            torch.cuda.synchronize()
            graph_ms = e0.elapsed_time(e1) / reps
            del graphs
        if int(status[0].item()):
            raise RuntimeError(f"device reported data errors (status {int(status[0].item()):#x}) in workload {cfg}/{B}")

        vb = float(np.mean([verify_bytes(sh) for sh in shapes]))
        cb = float(np.mean([commit_bytes(sh) for sh in shapes]))
        fb = float(np.mean([fused_bytes(sh) for sh in shapes]))
        T = float(np.mean([sh.T for sh in shapes]))
        pk = peaks["hbm_gbs"]
        gbs = lambda b, ms: b / (ms * 1e6)
        key = f"{WORKLOAD_NAMES[cfg][0]}_B{B}"
        out[key] = {
            "workload": workload_name(cfg, B), "layers_rotated": nl, "node_rows": T, "reps": reps,
            "l2": (f"flushed: {FLUSH_BYTES >> 20} MB scratch write before each pass (working set {ws / 2 ** 20:.0f} MB "
                   f"< 4x L2)") if flush else f"rotated: working set {ws / 2 ** 20:.0f} MB >= 4x L2",
            "verify_ms": v_ms, "commit_ms": c_ms, "step_ms": v_ms + c_ms, "fused_ms": f_ms,
            "eager_step_ms_back_to_back": eager_ms, "graph_step_ms": graph_ms,
            "verify_frac": gbs(vb, v_ms) / pk, "commit_frac": gbs(cb, c_ms) / pk,
            "step_frac": gbs(vb + cb, v_ms + c_ms) / pk, "fused_frac": gbs(fb, f_ms) / pk,
            "step_frac_of_nominal": gbs(vb + cb, v_ms + c_ms) / NOMINAL_HBM_GBS,
            "node_verifications_per_s": T / ((v_ms + c_ms) / 1e3),
            "node_verifications_per_s_fused": T / (f_ms / 1e3),
        }
        del layers, outs
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, "nccl")

    from gated_deltanet_tree_03_b300 import binding as gb
    from gated_deltanet_tree_03_b300 import device as gd

    layers = make_layers(args.config, args.batch, shard_layers(rank, args.layers))
    tb0 = layers[0]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(tb0)

    verify_fn = {"wy": gb.gdn_tree_verify, "simt": gb.gdn_tree_verify_simt}[args.kernel]
    dev_in = [gd.upload(tb, device=dev) for tb in layers]
    dev_out = [gd.alloc_outputs(tb, device=dev) for tb in layers]
    stream = torch.cuda.current_stream(dev)

    def step(i):
        tb, d, o = layers[i % len(layers)], dev_in[i % len(layers)], dev_out[i % len(layers)]
        verify_fn(d["ST"], d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"], d["cu_nodes"], tb.B, tb.H,
                  tb.T, tb.dk, tb.dv, tb.max_nodes, o["o"], o["U"], o["G"], o["status"], stream)
        return tb, d, o

    def commit(tb, d, o):
        gb.gdn_tree_commit(d["ST"], o["U"], o["G"], d["k"], d["parent"], d["cu_nodes"], d["path"], d["path_len"],
                           tb.B, tb.H, tb.T, tb.dk, tb.dv, tb.max_path, o["status"], stream)

    for i in range(args.warmup):
        commit(*step(i))
    torch.cuda.synchronize()
    status = sum(int(o["status"][0].item()) for o in dev_out)
    if status:
        raise RuntimeError(f"device reported data errors (status bits {status:#x})")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    t_wall = time.perf_counter()
    for i in range(K):
        ev[i][0].record(stream)
        tb, d, o = step(i)
        ev[i][1].record(stream)
        commit(tb, d, o)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    # the per-kernel breakdown takes its own repeat count (independent of --steps)
    Kr = max(1, args.kernel_reps)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Kr)]
    for i in range(Kr):
        kev[i][0].record(stream)
        tb, d, o = step(i)
        kev[i][1].record(stream)
        commit(tb, d, o)
        kev[i][2].record(stream)
    torch.cuda.synchronize()
    t_ver = sum(kev[i][0].elapsed_time(kev[i][1]) for i in range(Kr))
    t_com = sum(kev[i][1].elapsed_time(kev[i][2]) for i in range(Kr))
    total_ms = max_over_ranks(dist, total_ms, dev)
    nodes_per_step = tb0.T  # draft nodes of one layer's batch, all heads
    value = nodes_per_step * world * K / (total_ms / 1e3)

    # the same step replayed from CUDA graphs: each layer's verify + commit captured once (after the
    # warm-up, so every kernel is loaded), which removes the per-call host work from the step
    graph_step = None

    def time_graphs():
        graphs = []
        for j in range(len(layers)):
            tb, d, o = layers[j], dev_in[j], dev_out[j]
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                cs = torch.cuda.current_stream()
                verify_fn(d["ST"], d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"], d["cu_nodes"], tb.B,
                          tb.H, tb.T, tb.dk, tb.dv, tb.max_nodes, o["o"], o["U"], o["G"], o["status"], cs)
                gb.gdn_tree_commit(d["ST"], o["U"], o["G"], d["k"], d["parent"], d["cu_nodes"], d["path"],
                                   d["path_len"], tb.B, tb.H, tb.T, tb.dk, tb.dv, tb.max_path, o["status"], cs)
            graphs.append(gr)
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for i in range(K):
            graphs[i % len(graphs)].replay()
        g1.record()
        torch.cuda.synchronize()
        if sum(int(o["status"][0].item()) for o in dev_out):
            raise RuntimeError("device reported data errors in the graph replays")
        g_ms = max_over_ranks(dist, g0.elapsed_time(g1), dev) / K
        return {"value": tb0.T * world / (g_ms / 1e3), "unit": UNIT, "ms_per_step": g_ms, "steps": K,
                "gpu_launches": 2 * K,
                "note": "each layer's verify + commit captured once in a CUDA graph and replayed"}

    if args.graph:
        try:
            graph_step = time_graphs()
        except Exception as e:  # a capture this host cannot make is reported, not fatal
            graph_step = {"error": f"{type(e).__name__}: {e}"[:300]}

    peaks = measured_peaks()
    vb = float(np.mean([verify_bytes(tb) for tb in layers]))
    cb = float(np.mean([commit_bytes(tb) for tb in layers]))
    v_ms, c_ms = t_ver / Kr, t_com / Kr
    kernels = {
        "reps": Kr,
        "verify": {"ms": v_ms, "alg_bytes": vb, "GB/s": vb / (v_ms * 1e6), "frac": vb / (v_ms * 1e6) / peaks["hbm_gbs"]},
        "commit": {"ms": c_ms, "alg_bytes": cb, "GB/s": cb / (c_ms * 1e6), "frac": cb / (c_ms * 1e6) / peaks["hbm_gbs"]},
        "verify+commit": {"ms": v_ms + c_ms, "GB/s": (vb + cb) / ((v_ms + c_ms) * 1e6),
                          "frac": (vb + cb) / ((v_ms + c_ms) * 1e6) / peaks["hbm_gbs"]},
    }
    if args.fused:
        # deferred commit: every step commits the previous step's accepted paths and verifies the
        # next trees in one gdn_tree_commit_verify call (same inputs on both sides of the step;
        # the previous step's pseudo-values and log-gates alternate between two buffers per layer)
        nl = len(layers)
        pv = [[(torch.empty_like(o["U"]), torch.empty_like(o["G"])) for _ in range(2)] for o in dev_out]
        for j in range(nl):
            tb, d, o = layers[j], dev_in[j], dev_out[j]
            gb.gdn_tree_verify(d["ST"], d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"], d["cu_nodes"], tb.B,
                               tb.H, tb.T, tb.dk, tb.dv, tb.max_nodes, o["o"], pv[j][0][0], pv[j][0][1], o["status"],
                               stream)
        cur = [0] * nl

        def fused_step(i):
            j = i % nl
            tb, d, o = layers[j], dev_in[j], dev_out[j]
            (Up, Gp), (Un, Gn) = pv[j][cur[j]], pv[j][1 - cur[j]]
            gb.gdn_tree_commit_verify(d["ST"], Up, Gp, d["k"], d["parent"], d["cu_nodes"], d["path"], d["path_len"],
                                      tb.T, tb.max_path, d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"],
                                      d["cu_nodes"], tb.B, tb.H, tb.T, tb.dk, tb.dv, tb.max_nodes, o["o"], Un, Gn,
                                      o["status"], stream)
            cur[j] = 1 - cur[j]

        for i in range(args.warmup):
            fused_step(i)
        torch.cuda.synchronize()
        if sum(int(o["status"][0].item()) for o in dev_out):
            raise RuntimeError("device reported data errors in the fused steps")
        if dist is not None:
            dist.barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(K):
            fused_step(i)
        f1.record(stream)
        torch.cuda.synchronize()
        f_ms = max_over_ranks(dist, f0.elapsed_time(f1), dev) / K
        fb = float(np.mean([fused_bytes(tb) for tb in layers]))
        kernels["commit_verify"] = {"ms": f_ms, "alg_bytes": fb, "GB/s": fb / (f_ms * 1e6),
                                    "frac": fb / (f_ms * 1e6) / peaks["hbm_gbs"],
                                    "node_verifications_per_s": nodes_per_step * world / (f_ms / 1e3)}
    for kd in kernels.values():
        if isinstance(kd, dict):
            kd["frac_of_nominal"] = kd["GB/s"] / NOMINAL_HBM_GBS
    dom = "verify" if v_ms >= c_ms else "commit"
    wl = workload_key(args.config, tb0.B)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["GB/s"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": kernels[dom]["frac"], "peak_source": peaks["source"],
                "traffic": ncu_traffic(dom, wl), "nominal_peak": NOMINAL_HBM_GBS,
                "frac_of_nominal": kernels[dom]["GB/s"] / NOMINAL_HBM_GBS}

    # the store-all comparison the TreeWY page measures against: every node's state written
    # (T x H x d_k x d_v fp32 of snapshots per layer), commit = copy of the accepted one
    storeall = None
    if args.storeall:
        tb, d, o = layers[0], dev_in[0], dev_out[0]
        snap = torch.empty((tb.T, tb.H, tb.dk, tb.dv), device=dev)
        st_sa = torch.zeros(4, dtype=torch.int32, device=dev)

        def sa_verify():
            gb.gdn_tree_verify_storeall(d["ST"], d["q"], d["k"], d["v"], d["beta"], d["g"], d["parent"],
                                        d["cu_nodes"], tb.B, tb.H, tb.T, tb.dk, tb.dv, tb.max_nodes, snap, o["o"],
                                        o["U"], o["G"], st_sa, stream)

        def sa_commit():
            gb.gdn_tree_commit_storeall(d["ST"], snap, d["parent"], d["cu_nodes"], d["path"], d["path_len"], tb.B,
                                        tb.H, tb.T, tb.dk, tb.dv, tb.max_path, st_sa, stream)

        for _ in range(3):
            sa_verify()
            sa_commit()
        ns = 20
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        t_v = t_c = 0.0
        for _ in range(ns):
            evs[0].record(stream)
            sa_verify()
            evs[1].record(stream)
            sa_commit()
            evs[2].record(stream)
            torch.cuda.synchronize()
            t_v += evs[0].elapsed_time(evs[1])
            t_c += evs[1].elapsed_time(evs[2])
        if int(st_sa[0].item()):
            raise RuntimeError("device reported data errors in the store-all comparison")
        snap_bytes = snap.numel() * 4
        storeall = {"verify_ms": t_v / ns, "commit_ms": t_c / ns, "step_ms": (t_v + t_c) / ns,
                    "snapshot_bytes": snap_bytes,
                    "treewy_speculative_bytes": tb.T * tb.H * (tb.dv + 1) * 4,
                    "treewy_step_ms": v_ms + c_ms,
                    "note": "gdn_tree_verify_storeall + gdn_tree_commit_storeall on one layer of the same "
                            "workload; TreeWY keeps U and G (treewy_speculative_bytes) instead of every "
                            "node's state (snapshot_bytes)"}
        del snap

    # draft budgeting on the device: top-B positions (7 drafts per request, 3 per request on
    # average) and best-first growth over a ternary candidate tree of depth 7, at the batch size
    budget = None
    if args.budget:
        from gated_deltanet_tree_03_b300 import workloads as W
        rng = np.random.default_rng(77)
        R = tb0.B
        pa = torch.from_numpy(W.draw_acceptance(rng, R, 7)).to(dev)
        pe = torch.from_numpy(W.draw_edge_probs(rng, R, 3, 7)).to(dev)
        i32 = dict(dtype=torch.int32, device=dev)
        n_sel, cu_b, par_b = torch.empty(R, **i32), torch.empty(R + 1, **i32), torch.empty(R + 3 * R, **i32)
        n_g, pl_g = torch.empty(R, **i32), torch.empty(R * 64, **i32)
        cu_g, par_g = torch.empty(R + 1, **i32), torch.empty(R * 64, **i32)
        st_b = torch.zeros(4, **i32)
        calls = {"topb": lambda: gb.gdn_tree_budget_topb(pa, R, 7, 3 * R, n_sel, None, cu_b, par_b, st_b, stream),
                 "grow": lambda: gb.gdn_tree_grow_best_first(pe, R, 3, 7, 0.02, 64, n_g, pl_g, None, None, cu_g,
                                                             par_g, st_b, stream)}
        budget = {}
        for name, fn in calls.items():
            for _ in range(5):
                fn()
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            nb = 200
            b0.record(stream)
            for _ in range(nb):
                fn()
            b1.record(stream)
            torch.cuda.synchronize()
            budget[name] = {"ms": b0.elapsed_time(b1) / nb}
        if int(st_b[0].item()):
            raise RuntimeError("device reported data errors in the budget kernels")
        budget["topb"].update(requests=R, positions=7, budget=3 * R, launches=1,
                              selected=int(n_sel.sum().item()))
        budget["grow"].update(requests=R, fanout=3, depth=7, candidates=3280, threshold=0.02, max_nodes=64,
                              launches=2, mean_nodes=float(n_g.float().mean().item()))
        budget["note"] = ("latency-bound: one CTA sorts all R x 7 survival keys (top-B); one CTA per request sorts "
                          "its 3280 candidate keys (growth) plus one packing CTA; bytes moved are negligible")

    # tree-bias attention of the model's attention layers over the same kind of trees: 4096-key
    # committed prefixes, 16 query heads on 2 key/value heads, d = 128
    attention = None
    if args.attention:
        from gated_deltanet_tree_03_b300 import workloads as W
        attention = {}
        R = 64
        shapes = {"rootbranch6": [W.root_branch_parents()] * R,
                  "tree32": [W.random_tree_parents(np.random.default_rng(500 + i), 32, 3, 6) for i in range(R)]}
        for name, parents in shapes.items():
            ab = W.make_attention_batch(31, B=R, Hq=16, Hkv=2, d=128, prefix_range=(4096, 4096), parents=parents)
            bf = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
            i32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev)
            ins = [bf(ab.q), bf(ab.k), bf(ab.v), bf(ab.k_cache), bf(ab.v_cache), i32(ab.cu_prefix), i32(ab.parent),
                   i32(ab.cu_nodes)]
            o_a = torch.empty((ab.T, ab.Hq, ab.d), device=dev)
            wsb = gb.gdn_tree_attention_workspace_size(R, 16, 2, 128, ab.max_nodes, ab.max_prefix)
            ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
            st_a = torch.zeros(4, dtype=torch.int32, device=dev)
            fn = lambda: gb.gdn_tree_attention(*ins, R, 16, 2, ab.T, ab.P, 128, ab.max_nodes, ab.max_prefix, ab.scale,
                                               o_a, ws, wsb, st_a, stream)
            for _ in range(5):
                fn()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            na = 50
            a0.record(stream)
            for _ in range(na):
                fn()
            a1.record(stream)
            torch.cuda.synchronize()
            if int(st_a[0].item()):
                raise RuntimeError("device reported data errors in tree attention")
            ms = a0.elapsed_time(a1) / na
            ab_bytes, ab_flops = attention_bytes(ab), attention_flops(ab)
            attention[name] = {"ms": ms, "requests": R, "nodes": ab.T, "prefix_per_request": 4096, "heads_q": 16,
                               "heads_kv": 2, "d": 128, "workspace_bytes": wsb, "alg_bytes": ab_bytes,
                               "GB/s": ab_bytes / (ms * 1e6), "frac_hbm": ab_bytes / (ms * 1e6) / peaks["hbm_gbs"],
                               "useful_TFLOP/s": ab_flops / (ms * 1e9),
                               "frac_bf16": ab_flops / (ms * 1e9) / peaks["bf16_tflops"]}
            del ins, o_a, ws
        attention["note"] = ("gdn_tree_attention: each draft node attends to its request's committed prefix and "
                             "its own root-to-node path; K/V caches 268 MB (> L2); frac_hbm against the measured "
                             "copy bandwidth, frac_bf16 (useful flops) against the measured bf16 GEMM burst")

    # end to end: pinned host inputs -> device, verify + commit, outputs -> pinned host
    e2e = None
    if not args.no_e2e:
        keys = ["q", "k", "v", "beta", "g", "parent", "cu_nodes", "path", "path_len"]
        host_in = [gd.upload(tb, pin=True) for tb in layers]
        host_o = [torch.empty_like(o["o"], device="cpu").pin_memory() for o in dev_out]
        h2d = sum(host_in[0][k].numel() * host_in[0][k].element_size() for k in keys)
        d2h = host_o[0].numel() * host_o[0].element_size()
        Ke = max(1, min(K, args.e2e_steps))
        # three streams: copies in, the hot path, copies out; step i's inputs arrive while step i-1
        # runs and step i-1's outputs leave while step i runs. Each layer's buffers are reused only
        # after the step that last used them has finished with them.
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        nl = len(layers)
        comp_done = [None] * nl  # last hot-path event per layer (its inputs may be overwritten after)
        out_done = [None] * nl   # last copy-out event per layer (its o may be overwritten after)

        def e2e_step(i):
            j = i % nl
            with torch.cuda.stream(s_in):
                if comp_done[j] is not None:
                    s_in.wait_event(comp_done[j])
                for k in keys:
                    dev_in[j][k].copy_(host_in[j][k], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            stream.wait_event(ev_in)
            if out_done[j] is not None:
                stream.wait_event(out_done[j])
            commit(*step(i))
            ev_c = torch.cuda.Event()
            ev_c.record(stream)
            comp_done[j] = ev_c
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c)
                host_o[j].copy_(dev_out[j]["o"], non_blocking=True)
                ev_o = torch.cuda.Event()
                ev_o.record(s_out)
            out_done[j] = ev_o

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        stream.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(Ke):
            e2e_step(i)
        for ev in out_done:
            if ev is not None:
                s_in.wait_event(ev)
        e1.record(s_in)
        torch.cuda.synchronize()
        ems = max_over_ranks(dist, e0.elapsed_time(e1), dev)
        e2e = {"value": nodes_per_step * world * Ke / (ems / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": Ke,
               "note": "state resident in HBM across steps; every step copies its node block, tree and paths in "
                       "from pinned host memory and its o out, on copy streams overlapping the neighbouring steps"}

    workloads = None
    if args.workloads and world == 1:
        workloads = time_workloads(gb, dev, stream, peaks, args.kernel_reps)
    ws = sum(layer_bytes(tb) for tb in layers)
    l2 = (f"inputs larger than L2: {len(layers)} layers rotated, working set {ws / 2 ** 20:.0f} MB >= 4x L2"
          if ws >= 4 * L2_BYTES else f"working set {ws / 2 ** 20:.0f} MB below 4x L2 (L2-warm; not flushed)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_name(args.config, tb0.B), "batch_per_gpu": tb0.B, "heads": tb0.H,
                       "d_k": tb0.dk, "d_v": tb0.dv, "nodes_per_layer": nodes_per_step,
                       "layers_rotated": len(layers), "verify_kernel": args.kernel,
                       "l2": l2,
                       "parallelism": f"dp{world} (independent batches per GPU)"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 2 * K, "clocks": clk,
            "fused_commit_verify": None if "commit_verify" not in kernels else {
                "value": kernels["commit_verify"]["node_verifications_per_s"], "unit": UNIT,
                "ms_per_step": kernels["commit_verify"]["ms"], "achieved_GBps": kernels["commit_verify"]["GB/s"],
                "frac": kernels["commit_verify"]["frac"], "steps": K, "gpu_launches": K,
                "note": "gdn_tree_commit_verify: each step commits the previous step's accepted paths and verifies "
                        "the next trees in one pass over the state (deferred commit); same work as verify + commit"},
            "workloads": workloads, "graph_step": graph_step, "storeall": storeall, "tree_budget": budget, "tree_attention": attention, "kernels": kernels,
            "wall_s_timed": wall}
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--kernel", choices=["wy", "simt"], default="wy")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--ref-requests", type=int, default=1)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-storeall", dest="storeall", action="store_false",
                    help="skip timing the store-all comparison (every node's state written)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="skip timing the step replayed from CUDA graphs (which removes the per-call host work)")
    ap.add_argument("--no-attention", dest="attention", action="store_false",
                    help="skip timing tree-bias attention (gdn_tree_attention)")
    ap.add_argument("--no-budget", dest="budget", action="store_false",
                    help="skip timing the draft-budgeting kernels (top-B positions, best-first growth)")
    ap.add_argument("--kernel-reps", type=int, default=200,
                    help="passes behind the per-kernel breakdown and each workloads entry")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip timing every preset batch (the workloads object)")
    ap.add_argument("--no-fused", dest="fused", action="store_false",
                    help="skip timing gdn_tree_commit_verify (the previous step's commit folded into the next verify)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
