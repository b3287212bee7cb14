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


def _oracle_outputs(bt, mode):
    import torch
    import oracle
    p, q, t, ua, ur, md = bt.numpy()
    if mode == "greedy":
        n, x, _ = oracle.verify_greedy(p, t)
    elif mode == "sample":
        n, x, _ = oracle.verify_sample(p, q, t, ua, ur)
    else:
        n, x, _ = oracle.verify_round(md, p, q, t, ua, ur)
    return torch.from_numpy(np.array(n, dtype=np.int32)), torch.from_numpy(np.array(x, dtype=np.int32))


@pytest.mark.parametrize("mode,cfg", [("sample", 3), ("greedy", 2), ("round", 4)])
def test_bench_parity_leg_counts_and_takes_bytes_from_the_oracle(mode, cfg):
    """The CPU-baseline leg's parity check: outputs equal to the oracle's give
    no mismatch and the oracle's required bytes; one planted wrong token is a
    decision mismatch, not a boundary case."""
    from speculative_decoding_verification_08_gb300.inputs import make_inputs
    sets = [make_inputs(cfg, "cpu", seed=77 + i, B=12, V=700, K=4) for i in range(2)]
    outs = [_oracle_outputs(bt, mode) for bt in sets]
    par, req = bench.oracle_parity(sets, outs, [], mode, 4, 700)
    assert par["sets"] == 2 and par["sequences"] == 24
    assert par["decision_mismatches"] == 0 and par["boundary_mismatches"] == 0
    for bt, (n, _), r in zip(sets, outs, req):
        md = (np.zeros(12) if mode == "greedy" else np.ones(12) if mode == "sample"
              else bt.mode.numpy())
        assert r == bench.required_bytes(md, n.numpy(), 4, 700)
    n, x = outs[1]
    x[3] = (x[3] + 1) % 700 if x[3] >= 0 else 5   # a token the oracle did not draw
    par, _ = bench.oracle_parity(sets, outs, [], mode, 4, 700)
    assert par["decision_mismatches"] == 1
