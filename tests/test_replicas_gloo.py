"""The multi-GPU path is replicas only (tokens shard across ranks, no
collective on the data path).  This runs bench.py's rank bookkeeping -- the
barrier and the max-over-ranks step time -- as two gloo ranks on the CPU, and
checks that every replica draws its own batch."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    from group_limited_routing_gb300 import workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = bench.max_over_ranks(world, 1.0 + rank, "cpu")
        w0 = wl.WORKLOADS[1]
        x = wl.hidden(w0, "cpu", layer=rank) if rank else wl.hidden(w0, "cpu")
        digest = float(x.float().sum())
        bench.barrier(world)
        q.put((rank, ms, digest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_agree_on_the_max_step_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [2.0, 2.0]          # every rank reports the slowest rank's time
    assert res[0][2] != res[1][2]                      # each replica its own batch
