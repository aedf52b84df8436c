"""The N > 1 host path of bench.py (weak scaling, max-over-ranks timing) on gloo ranks."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = [7.0, 11.0, 5.0, 9.0][rank]
    ms = bench.reduce_max(ms_local)
    v = bench.whole_job_value(4096 * 4096, world, ms)
    q.put((rank, ms, v))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_max_over_ranks_and_weak_scaling(world):
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
    expect = max([7.0, 11.0, 5.0, 9.0][:world])
    for _, ms, v in res:
        assert ms == expect
        assert v == pytest.approx(world * 4096 * 4096 / (expect / 1e3))


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
