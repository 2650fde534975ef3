"""The multi-GPU path of the benchmark is replicas only: each rank runs its own
batch, and only the timing scalars cross ranks.  Two gloo ranks on the CPU
check the barrier, the max over ranks and the weak-scaling throughput."""
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
                      WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench._barrier(world)
        ms_local = 10.0 + 5.0 * rank          # rank 1 is the slow one
        ms_max = bench._max_over_ranks(ms_local, world, "cpu")
        q.put((rank, ms_max, bench.job_throughput(256, world, ms_max)))
        bench._barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms_max, value in got:
        assert ms_max == 15.0
        assert value == pytest.approx(256 * 2 / 15e-3)
