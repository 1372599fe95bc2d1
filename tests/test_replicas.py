"""The multi-GPU path is replicas only: each rank runs its own copy of the
workload with no collective on the data path; the host takes the slowest
rank's time and reports the bytes of all ranks over it.  That host logic runs
here on CPU with two gloo ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, elapsed, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    e = bench.max_over_ranks(elapsed[rank], world)
    out[rank] = (e, bench.whole_job_gbs(1_000_000, 50, world, e))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        elapsed = [0.010, 0.025]
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, elapsed, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            e, gbs = out[r]
            assert e == pytest.approx(0.025)
            assert gbs == pytest.approx(2 * 1_000_000 * 50 / 0.025 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.whole_job_gbs(2_000_000_000, 1, 1, 1.0) == pytest.approx(2.0)
