"""The multi-rank timing logic of bench.py on CPU (gloo, world size 2): each
rank reports its own device time, the job time is the max over ranks, and the
whole-job value counts the work of every rank."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [100.0, 250.0][rank]
        m = bench.max_over_ranks(local_ms)
        v = bench.aggregate_tflops(1e12, world, m, 10)
        q.put((rank, m, v, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v, env in out:
        assert m == 250.0
        # 2 ranks x 10 steps x 1 TFLOP over 0.25 s
        assert v == pytest.approx(2 * 10 * 1.0 / 0.25)
        assert env[0] == rank and env[1] == 2


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate_tflops(2e12, 1, 1000.0, 4) == pytest.approx(8.0)
