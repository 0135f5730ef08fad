"""The N > 1 path of bench.py on CPU: two gloo ranks, each with its own
independent request, reduce to the slowest rank's time and the sum of tokens."""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    secs, toks = bench.aggregate(1.5 + rank, 10.0 * (rank + 1), world, "cpu")
    out[rank] = (secs, toks, bench.replica_seed(rank))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_tokens():
    ctx = mp.get_context("spawn")
    world = 2
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        assert res[r][0] == 2.5          # slowest rank
        assert res[r][1] == 30.0         # 10 + 20 tokens
    assert res[0][2] != res[1][2]        # each replica decodes its own request


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(3.0, 7.0, 1) == (3.0, 7.0)
