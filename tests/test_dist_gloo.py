"""The N > 1 bench path on CPU: two gloo ranks, replicas only.  The whole-job value is all ranks'
units over the slowest rank's time, and every rank agrees on it."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        seconds = 2.0 if rank == 1 else 1.0
        value, t = bench.aggregate(10.0, seconds, world)
        q.put((rank, value, t, bench.reduce_max(rank * 3.0)))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, t, mx in res:
        assert t == 2.0
        assert value == 2 * 10.0 / 2.0
        assert mx == 3.0


def test_single_process_identity():
    import bench
    assert bench.aggregate(6.0, 3.0, 1) == (2.0, 3.0)
