"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The verify/commit path has no data-path collective: each rank processes its own batches
(weak scaling), the step time is the maximum over ranks and the reported throughput counts
every rank's nodes. These tests run the benchmark's own helpers in two gloo ranks and check
that the ranks' input sets are disjoint, that the timing reduction is a max, and that the
per-rank work (checked here with the CPU oracle on each rank's shard) adds up to the whole.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    import bench
    import oracle
    from gated_deltanet_tree_03_b300 import workloads as W

    w, r, _ = bench.dist_env()
    assert (w, r) == (world, rank)
    d = bench.dist_init(w, "gloo")
    assert d is not None
    layers = bench.shard_layers(r, 3)
    # each rank's step time differs; the reported time is the max over ranks
    t = bench.max_over_ranks(d, 1.0 + rank, torch.device("cpu"))
    gathered = [None] * world
    dist.all_gather_object(gathered, layers)
    # per-rank work: a small tree batch per input set, verified by the oracle on that rank
    nodes = 0
    for layer in layers:
        tb = W.make_random_batch(seed=1000 + layer, B=2, H=2, d=16, n_range=(2, 6))
        inp = oracle.batch_inputs(tb)
        o, U, G = oracle.verify(**inp)
        assert np.all(np.isfinite(o))
        nodes += tb.T
    totals = [None] * world
    dist.all_gather_object(totals, nodes)
    np.save(os.path.join(out_dir, f"rank{rank}.npy"),
            np.array([t, sum(totals)] + [x for g in gathered for x in g], dtype=np.float64))
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_disjointly_and_time_by_max(tmp_path):
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [np.load(os.path.join(tmp_path, f"rank{r}.npy")) for r in range(world)]
    for r in range(world):
        t, total = res[r][0], res[r][1]
        assert t == float(world)  # max over ranks of 1 + rank
        layer_ids = res[r][2:].astype(int).tolist()
        assert len(layer_ids) == len(set(layer_ids)) == 3 * world  # disjoint input sets
    assert res[0][1] == res[1][1] > 0  # every rank agrees on the whole job's node count


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(None, 2.5, None) == 2.5
    assert bench.shard_layers(0, 4) == [0, 1, 2, 3]
    assert bench.shard_layers(1, 4) == [4, 5, 6, 7]
