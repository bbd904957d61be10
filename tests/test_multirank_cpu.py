"""The bench's multi-rank host logic on CPU: two gloo ranks, each running its
own batch, combine into whole-job figures (slowest rank's time, all ranks'
tokens) with no other collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import gdnsynth as sy
    ms, tok = bench.reduce_across_ranks(10.0 + rank, 100.0 * (rank + 1))
    spec = bench.rank_spec(sy.SPECS["paged256"], rank)
    out.put((rank, ms, tok, spec.seed))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [11.0, 11.0]          # max of the timed regions
    assert [r[2] for r in res] == [300.0, 300.0]        # sum of verified tokens
    assert res[0][3] != res[1][3]                       # each rank draws its own requests


def test_single_process_needs_no_group():
    import bench
    assert bench.reduce_across_ranks(5.0, 7.0) == (5.0, 7.0)
