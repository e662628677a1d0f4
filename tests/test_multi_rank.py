"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2).

Chains are independent, so N GPUs run N copies of the workload with no collective on
the data path. What remains on the host is checked here: each rank draws a distinct
seeded input set, and the reported time is the maximum over ranks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import kda_synth as S
    d = bench.init_dist(world, "gloo")
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        # each rank times something different; everyone must report the slowest
        t = bench.max_over_ranks(1.5 + rank, d)
        cfg = S.configs()["prefill_h1_t64"]
        inp = S.prefill_inputs(cfg.seqlens, cfg.num_heads, seed=bench.rank_seed(cfg.seed, rank), init_std=None)
        gathered = [torch.zeros_like(inp["q"]) for _ in range(world)]
        dist.all_gather(gathered, inp["q"])
        distinct = not torch.equal(gathered[0], gathered[1])
        results[rank] = (t, distinct)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_timing_and_distinct_inputs():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == 2.5
    assert res[0][1] and res[1][1]


def test_rank_seed_is_distinct_and_stable():
    import bench
    seeds = {bench.rank_seed(1, r) for r in range(8)}
    assert len(seeds) == 8 and bench.rank_seed(1, 0) == 1
