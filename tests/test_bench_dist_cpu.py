"""The bench's multi-rank path on CPU: two gloo ranks, max elapsed time and summed units.

bench.py runs N independent replicas (one per GPU) with no data-path collective; the only
cross-rank step is this aggregation of the timed region."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w, r, l = bench.dist_env()
        assert (w, r, l) == (world, rank, rank)
        t, u = bench.aggregate(0.5 + rank, 1000.0 * (rank + 1))
        bench.barrier()
        q.put((rank, t, u))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_aggregate_max_time_sum_units(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, u in res:
        assert t == 0.5 + (world - 1)
        assert u == sum(1000.0 * (r + 1) for r in range(world))


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(1.25, 7.0) == (1.25, 7.0)
