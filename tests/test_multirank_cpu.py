"""The bench's multi-rank logic on the CPU: two gloo ranks on 127.0.0.1.

Under torchrun each rank runs its own replica of the path (tokens are independent, so there is
no collective on the data path). What is shared is the timing: every rank's time is reduced to
the maximum, and the job's throughput is all ranks' units over that time. The reference arm
runs on rank 0 only; other ranks leave without printing.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t_max = bench.reduce_max(1.5 + rank, world, "cpu")
    rate = bench.job_rate(world, 100, t_max)
    dist.barrier()
    out = io.StringIO()
    if rank != 0:
        # the reference arm: only rank 0 works and prints
        class A:
            pass
        a = A()
        with redirect_stdout(out):
            bench.run_reference(a)
    dist.destroy_process_group()
    q.put((rank, t_max, rate, out.getvalue()))


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, rate, printed in res:
        assert t_max == 2.5                        # the slowest rank's time, on every rank
        assert rate == world * 100 / 2.5          # all ranks' units over that time
        if rank != 0:
            assert printed == ""                   # non-zero ranks print nothing


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25, 1, "cpu") == 3.25
    assert bench.job_rate(1, 64, 2.0) == 32.0
