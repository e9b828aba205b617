"""The multi-rank path of bench.py, on CPU with two gloo ranks.

Across GPUs the hot path runs as independent replicas: every rank processes
its own batch with no collective on the data path, and the only cross-rank
steps are the barriers around the timed region and the reduction of the
timing (slowest rank) and of the work done (sum over ranks) into one
whole-job figure.  These tests run exactly those host steps as two real
processes over gloo, with different work and time on each rank, including
the rule that only rank 0 of the reference arm does any work.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dev = torch.device("cpu")
        bench._barrier(True)
        # rank r processed 1000 * (r + 1) units in 10 * (r + 1) ms over 5 steps
        units, ms = 1000.0 * (rank + 1), 10.0 * (rank + 1)
        value, ms_step = bench.job_rate(units, ms, 5, True, dev)
        mx = bench._max_over_ranks(3.0 + rank, True, dev)
        sm = bench._sum_over_ranks(2.0 ** rank, True, dev)
        bench._barrier(True)

        class Args:
            steps, warmup, gpus = 1, 0, world
        ref = bench.reference_arm(Args, rank) if rank != 0 else "rank0-skipped"
        out[rank] = (value, ms_step, mx, sm, ref)
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    # units summed over ranks (1000 + 2000), time of the slowest rank (20 ms over 5 steps)
    for r in range(world):
        value, ms_step, mx, sm, _ = res[r]
        assert ms_step == pytest.approx(4.0)
        assert value == pytest.approx(3000.0 / 4e-3)
        assert mx == 4.0 and sm == 3.0
    # the reference arm: every rank but 0 exits without work
    assert res[1][4] is None


def test_single_rank_needs_no_process_group():
    import bench
    value, ms_step = bench.job_rate(500.0, 20.0, 4, False, torch.device("cpu"))
    assert ms_step == pytest.approx(5.0) and value == pytest.approx(500.0 / 5e-3)
    assert bench._max_over_ranks(7.0, False, None) == 7.0


def _head_shard_worker(rank, world, port, out):
    """Rank r runs the oracle prefill on its contiguous share of the heads and of the groups
    (tensor parallelism splits nheads and ngroups together), then the shares are gathered."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np
        import oracle
        rng = np.random.default_rng(41)
        T, H, P, N, G = 90, 4, 4, 6, 2
        cu, cc = [0, 37, 90], [0, 16, 37, 53, 69, 85, 90]
        x, dt = rng.standard_normal((T, H, P)), rng.standard_normal((T, H))
        B, C = rng.standard_normal((T, G, N)), rng.standard_normal((T, G, N))
        A, D, bias = -np.exp(rng.uniform(0, 2, H)), rng.standard_normal(H), rng.uniform(-4, -1, H)
        h0 = rng.standard_normal((2, H, P, N))
        hs = slice(rank * H // world, (rank + 1) * H // world)
        gs = slice(rank * G // world, (rank + 1) * G // world)
        y, cs, fs = oracle.ssd_prefill(x[:, hs], dt[:, hs], A[hs], B[:, gs], C[:, gs], cu, cc, D=D[hs],
                                       dt_bias=bias[hs], initial_states=h0[:, hs])
        parts = [None] * world
        dist.all_gather_object(parts, (y, cs, fs))
        if rank == 0:
            full = oracle.ssd_prefill(x, dt, A, B, C, cu, cc, D=D, dt_bias=bias, initial_states=h0)
            got = [np.concatenate([p[i] for p in parts], axis=1) for i in range(3)]
            out[0] = all(np.array_equal(g, f) for g, f in zip(got, full))
    finally:
        dist.destroy_process_group()


def test_heads_shard_across_two_gloo_ranks_without_exchange():
    """The path shards by heads: two ranks, each with half the heads and the groups those heads
    use, and no data exchanged between them, reproduce the single-rank outputs, chunk states and
    final states bit for bit (the union of the shares is the whole result)."""
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_head_shard_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        assert out[0] is True
