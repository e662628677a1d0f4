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


CHILD = r'''
import json, os, sys
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_env()
if os.environ.get("FAIL_RANK") == str(rank):
    sys.exit(3)
d = bench.init_dist(world, "gloo")
t = bench.max_over_ranks(10.0 + rank, d)
d.barrier()
if rank == 0:
    print(json.dumps({{"world": world, "max": t, "local": local, "addr": os.environ["MASTER_ADDR"]}}), flush=True)
d.destroy_process_group()
'''


@pytest.mark.timeout(180)
def test_gpus_flag_launches_replicas_itself(tmp_path, capfd):
    """bench.py --gpus N outside torchrun starts N rank processes with the torchrun environment;
    rank 0 alone prints, with the maximum over ranks."""
    import json

    import bench
    script = tmp_path / "child.py"
    script.write_text(CHILD.format(root=bench.ROOT))
    import sys
    rc = bench.launch_replicas(2, [], cmd=[sys.executable, str(script)], timeout_s=150)
    out = capfd.readouterr().out.strip().splitlines()
    assert rc == 0
    lines = [json.loads(x) for x in out if x.startswith("{")]
    assert lines == [{"world": 2, "max": 11.0, "local": 0, "addr": "127.0.0.1"}]


@pytest.mark.timeout(180)
def test_replica_launcher_stops_the_job_when_a_rank_fails(tmp_path, monkeypatch):
    """A rank that exits with an error ends the job with its code; the rank left waiting in the
    rendezvous is stopped instead of hanging."""
    import sys

    import bench
    script = tmp_path / "child.py"
    script.write_text(CHILD.format(root=bench.ROOT))
    monkeypatch.setenv("FAIL_RANK", "1")
    rc = bench.launch_replicas(2, [], cmd=[sys.executable, str(script)], timeout_s=150)
    assert rc == 3
