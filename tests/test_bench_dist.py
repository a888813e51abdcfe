"""The benchmark's multi-rank host logic on CPU: replicas report their IDs and
elapsed time, and the whole-job figures are the sum of IDs and the maximum
time over ranks (gloo, world size 2; no GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ids, secs = bench.aggregate(1000.0 * (rank + 1), 0.5 + rank)
    q.put((rank, ids, secs))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_aggregate_sums_ids_and_takes_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=90) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, ids, secs in out:
        assert ids == 3000.0 and secs == 1.5


def test_aggregate_single_process_is_identity():
    import bench
    assert bench.aggregate(123.0, 0.25) == (123.0, 0.25)
