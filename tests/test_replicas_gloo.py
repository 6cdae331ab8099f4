"""The N>1 path of bench.py on CPU: world_size-2 gloo ranks.

Sequences are independent and the weights are replicated, so N GPUs run N
independent replicas of the round, with no collective on the data path (weak
scaling).  What the N>1 path adds on the host is checked here with two real
processes: each rank draws its own seeded batch, the timings are reduced with a
max over ranks, and the whole-job rate counts every rank's draft tokens.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from pe_workload import config, make_round


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = config(0)
        seed = bench.replica_seed(cfg.seed, rank, world)
        rnd = make_round(cfg, seed)
        # every rank's own batch, gathered only to check independence
        mine = torch.from_numpy(np.ascontiguousarray(rnd.prev_tokens, dtype=np.int64)).flatten()
        gathered = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(gathered, mine)
        ms = [1.0 + rank, 5.0 - rank]  # per-rank timings (ms): the job's time is the max over ranks
        red = bench.max_over_ranks(ms, dist, "cpu")
        out[rank] = dict(seed=seed, distinct=not torch.equal(gathered[0], gathered[1]), red=red,
                         rate=bench.whole_job_rate(world, cfg.B, cfg.K, red[0]))
    finally:
        dist.destroy_process_group()


def test_two_replicas_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    cfg = config(0)
    assert res[0]["seed"] == cfg.seed and res[1]["seed"] == cfg.seed + 1000
    assert res[0]["distinct"] and res[1]["distinct"]          # independent replicas
    assert res[0]["red"] == res[1]["red"] == [2.0, 5.0]       # max over ranks on every rank
    assert res[0]["rate"] == pytest.approx(world * cfg.B * cfg.K / 2.0e-3)


def test_single_rank_is_the_plain_workload():
    cfg = config(1)
    assert bench.replica_seed(cfg.seed, 0, 1) == cfg.seed
    assert bench.max_over_ranks([3.0, 4.0], None, "cpu") == [3.0, 4.0]
    assert bench.whole_job_rate(1, cfg.B, cfg.K, 0.25) == pytest.approx(cfg.B * cfg.K / 0.25e-3)
