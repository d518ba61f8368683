"""The multi-rank host path of bench.py on CPU: two gloo ranks.

Under torchrun every rank runs its own layer calls on its own tokens against
replicated weights (weak scaling, no exchange on the data path).  These
tests check what that needs: each rank's activations are a distinct,
reproducible piece of one global token stream, the timing reduction takes
the slowest rank, and a rank's outputs (here from the oracle) are the rows
the single-rank run gives for the same tokens.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import workloads

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, cfg, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = bench.rank_tokens(cfg, rank, world)
        # disjoint and complete: gather every rank's tokens
        mine = torch.from_numpy(x.astype(np.int32))
        allx = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(allx, mine)
        # the slowest rank's time
        slowest = bench.max_over_ranks(1.0 + rank, world)
        # one call of this rank through the oracle (token rows are independent)
        layer = workloads.make_layer(cfg)
        out = oracle.moe_forward(x[:cfg.T], layer, keep_intermediates=False).out
        results[rank] = (np.stack([a.numpy() for a in allx]), slowest, out)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_shard_the_token_stream():
    cfg = workloads.CONFIGS["tiny"].scaled(calls=3)
    port = _free_port()
    with mp.Manager() as man:
        results = man.dict()
        mp.spawn(_worker, args=(WORLD, port, cfg, results), nprocs=WORLD, join=True)
        res = dict(results)
    whole = workloads.normal_bf16(0, workloads.STREAM_X, (WORLD * cfg.calls * cfg.T, cfg.H),
                                  cfg.x_std)
    per = cfg.calls * cfg.T
    for rank in range(WORLD):
        gathered, slowest, out = res[rank]
        assert slowest == float(WORLD)
        for r in range(WORLD):
            # rank r's tokens are rows [r*per, (r+1)*per) of the global stream
            assert np.array_equal(gathered[r].astype(np.uint16), whole[r * per:(r + 1) * per])
        # the rank's first call equals the single-rank oracle on those rows
        ref = oracle.moe_forward(whole[rank * per:rank * per + cfg.T], workloads.make_layer(cfg),
                                 keep_intermediates=False).out
        np.testing.assert_array_equal(out, ref)


def test_single_rank_is_the_whole_stream():
    cfg = workloads.CONFIGS["tiny"].scaled(calls=2)
    x = bench.rank_tokens(cfg, 0, 1)
    whole = workloads.normal_bf16(0, workloads.STREAM_X, (cfg.calls * cfg.T, cfg.H), cfg.x_std)
    assert np.array_equal(x, whole)
    assert bench.max_over_ranks(2.5, 1) == 2.5


def _health_worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from sparse_moe_expert_gb300.health import ExpertHealthMonitor

        def accumulate(counts, window):
            window += counts.to(torch.int64)

        def reduce(window):
            return oracle.expert_health(window.numpy())

        mon = ExpertHealthMonitor(6, "cpu", clock=lambda: 0.0, accumulate=accumulate,
                                  reduce=reduce, process_group=dist.group.WORLD)
        rng = np.random.default_rng(100 + rank)
        mine = np.zeros(6, np.int64)
        for _ in range(3):
            c = rng.integers(0, 20, 6).astype(np.int32)
            mine += c
            mon.record(torch.from_numpy(c))
        h = mon.close_window()
        results[rank] = (mine, (h.least_expert, h.mean, h.std))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_health_window_sums_the_ranks():
    """With a process group each rank's closed window reports the health of
    the counts of all ranks together."""
    port = _free_port()
    with mp.Manager() as man:
        results = man.dict()
        mp.spawn(_health_worker, args=(WORLD, port, results), nprocs=WORLD, join=True)
        res = dict(results)
    total = sum(res[r][0] for r in range(WORLD))
    want = oracle.expert_health(total)
    for r in range(WORLD):
        assert res[r][1] == want
