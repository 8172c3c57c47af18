"""bench.py's multi-rank host logic on CPU with two gloo ranks.

The path shards by batch with no exchange step, so several GPUs run
independent replicas; the only cross-rank operation is the max of the ranks'
timings.  These tests run that reduction over a real gloo process group.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([10.0 * (rank + 1), 3.0 - rank], world)
    out_q.put((rank, got, bench.whole_job_us_per_layer(got[0], 100, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, us in res:
        assert got == [20.0, 3.0]          # the slowest rank's time for each value
        assert us == pytest.approx(20.0 * 1e3 / (100 * 2))


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.whole_job_us_per_layer(2.0, 4, 1) == pytest.approx(500.0)
