"""Host logic of the multi-GPU bench path (replicas, no data-path collective),
exercised with world_size 2 over gloo on the CPU: per-rank token seeds, the
max-over-ranks timing reduction and the whole-job aggregation."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, _ = bench.dist_env()
    # each rank times a different amount; the job time is the slowest rank's
    mine = [10.0 + rank, 20.0 - rank, 1.5 * (rank + 1)]
    got = bench.max_over_ranks(mine, dist, "cpu")
    seeds = [bench.rank_token_seed(0, i) for i in range(world)]
    dist.barrier()
    q.put((r, w, got, seeds))
    dist.destroy_process_group()


def test_two_rank_timing_reduction_and_seeds():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, got, seeds in res:
        assert w == world
        assert got == [11.0, 20.0, 3.0]
        assert len(set(seeds)) == world and seeds[0] == 0


def test_aggregate_throughput_is_whole_job():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    tf, tok = bench.aggregate_throughput(1e12, 1000, 4, 2.0)
    assert tf == pytest.approx(4 * 1e12 / 2e-3 / 1e12)
    assert tok == pytest.approx(4 * 1000 / 2e-3)
