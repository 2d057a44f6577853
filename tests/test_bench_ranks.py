"""The multi-rank bench logic on CPU: two gloo ranks run replicas; the job time is the slowest
rank's and the token count the sum of all ranks'."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [12.5, 20.0][rank]
    toks = [70, 70][rank]
    q.put((rank, bench.reduce_over_ranks(ms, toks, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == (20.0, 140) and res[1] == (20.0, 140)


def test_single_rank_passthrough():
    import bench
    assert bench.reduce_over_ranks(3.0, 7, 1) == (3.0, 7)
