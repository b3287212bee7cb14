"""Host-side logic of bench.py: required-bytes accounting, per-rank seeds and
the max-over-ranks timing reduction on a world-size-2 gloo group (CPU)."""
import os

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_required_bytes_follow_the_rule():
    K, V = 5, 1000
    # greedy: rows 0..n
    assert bench.required_bytes([0], [0], K, V) == 4 * V + 4 * K + 8
    assert bench.required_bytes([0], [K], K, V) == (K + 1) * 4 * V + 4 * K + 8
    # sampling: a rejected sequence reads the row pair, an accepted one p_K only
    rej = bench.required_bytes([1], [2], K, V)
    acc = bench.required_bytes([1], [K], K, V)
    assert rej == 64 * 3 + 8 * V + 8 * K + 16
    assert acc == 64 * K + 4 * V + 8 * K + 16
    assert bench.dense_bytes([1, 0], K, V) == 2 * (K + 1) * 4 * V + K * 4 * V


def test_rank_seeds_are_distinct():
    seeds = {bench.rank_seed(3, s, r) for s in range(4) for r in range(8)}
    assert len(seeds) == 32


def test_args_defaults_and_checks():
    a = bench.parse_args([])
    assert a.config == 3 and a.mode == "sample" and a.steps > 0 and a.warmup >= 3
    assert bench.parse_args(["--config", "2"]).mode == "greedy"
    assert bench.parse_args(["--config", "4"]).mode == "round"
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "1"])


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.reduce_max(10.0 + rank * 5.0)
        bench.barrier()
        v = bench.aggregate_rounds_per_s(1000, world, m / 1000.0)
        out[rank] = (m, v)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    port = 29500 + (os.getpid() % 2000)
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert np.isclose(res[0][1], 1000 * 2 / 0.015)


def test_trace_flag_parses():
    import bench
    a = bench.parse_args(["--trace", "--mode", "greedy"])
    assert a.trace and a.mode == "greedy"
    assert not bench.parse_args([]).trace
