"""The multi-rank logic of bench.py on CPU: two gloo ranks, no GPU.  The method has no
exchange step, so N ranks run independent replicas; what needs checking is the request
sharding (every request served exactly once when there are enough requests, replicas when
there are fewer) and the max-over-ranks step time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        t = bench.max_over_ranks(1.5 + rank, world)
        bench.barrier(world)
        out[rank] = {"max": t, "shard4": bench.shard_requests(4, rank, world),
                     "shard1": bench.shard_requests(1, rank, world)}
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0]["max"] == res[1]["max"] == 2.5
    assert sorted(res[0]["shard4"] + res[1]["shard4"]) == [0, 1, 2, 3]
    assert res[0]["shard1"] == res[1]["shard1"] == [0]
