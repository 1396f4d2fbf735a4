"""The multi-GPU form of the benchmark is replicas only (groups are independent, and
one batch has no exchange step): each rank runs its own copy, and the job's rate is
every rank's work over the slowest rank's time.  The host side of that path - the
max-over-ranks reduction and the whole-job rate - runs here on CPU with two gloo
ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [120.0, 150.0][rank]
    rate, ms = bench.replica_throughput(1e12, ms_local, world)
    q.put((rank, rate, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replica_throughput_uses_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rate, ms in got:
        assert ms == 150.0
        assert abs(rate - 2e12 / 0.150) < 1e-3 * rate


def test_single_process_is_the_identity():
    import bench
    rate, ms = bench.replica_throughput(5e11, 100.0, 1)
    assert ms == 100.0 and abs(rate - 5e12) < 1e-6 * rate
