"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2): each rank
runs an independent replica on its own store (distinct seeds); the timing is
the max over ranks and the token count the sum, with no data-path collective."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

_ENV_BEFORE = {v for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
               if os.environ.get(v) == "1"}


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


def test_oracle_pool_counts_every_step_once():
    """The CPU baseline's process pool runs exactly the steps it is given and
    sums the tokens of all workers (tiny workload, 2 spawned workers)."""
    import bench
    from synth import workloads
    wl = workloads.get("tiny")
    cache = bench._host_cache(wl)()
    per_step = bench.oracle_step(wl, 0, 4, lambda: cache)
    run = bench.oracle_pool(wl.spec, 4, 2, [3, 2], warmup=1)
    assert run["reps"] == 5
    assert run["tokens"] == 5 * per_step
    assert run["wall_s"] > 0 and run["value"] == run["tokens"] / run["wall_s"]
    for v in bench._ONE_THREAD:                  # the parent's environment is restored
        assert os.environ.get(v) != "1" or v in _ENV_BEFORE
