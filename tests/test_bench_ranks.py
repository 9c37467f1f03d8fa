"""The benchmark's multi-rank path on CPU: two gloo ranks, each timing its own
replica; the reported time is the max over ranks and the work the sum."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env()[:2] == (world, rank)
    bench.barrier(world)
    t, u = bench.aggregate(10.0 + 5.0 * rank, 100.0 * (rank + 1), world)
    out[rank] = (t, u)
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (15.0, 300.0)


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)
