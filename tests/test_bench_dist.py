"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2): each rank
runs an independent replica on its own store (distinct seeds); the timing is
the max over ranks and the token count the sum, with no data-path collective."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        assert bench.dist_env()[:2] == (rank, world)
        t = bench.reduce_max(1.5 + rank)          # per-rank elapsed ms
        n = bench.reduce_sum(1000.0 * (rank + 1))  # per-rank tokens
        bench.barrier()
        out[rank] = (t, n, bench.rank_seed(2, rank))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_and_distinct_seeds():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5
    assert res[0][1] == res[1][1] == 3000.0
    assert res[0][2] != res[1][2]
