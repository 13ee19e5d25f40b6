"""The multi-GPU form of the benchmark is replicas only (tokens shard with no
exchange step): each rank times its own copy of the workload, ranks meet at
a barrier on both sides of the timed region and the slowest rank's time is
reported. These helpers are checked here with two gloo ranks on the CPU."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        mx = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")
        bench.rank_barrier(world)
        results[rank] = mx
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(results) == {0: 20.0, 1: 20.0}


def test_single_rank_helpers_are_identity():
    import bench
    bench.rank_barrier(1)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
