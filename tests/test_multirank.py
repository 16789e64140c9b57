"""The multi-rank host logic of bench.py on CPU ranks (gloo, world size 2): every rank runs its
own copy of the workload (the heads of a problem are independent, so there is no data-path
collective), the job's time is the slowest rank's, and the whole-job rate counts every rank's
work.  No GPU is involved."""
import datetime
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    # a bounded rendezvous and collectives: a rank that never arrives fails the test instead of
    # hanging it (whether or not the pytest-timeout plugin is installed)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=60))
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms)
        value = bench.whole_job_tflops(2.0e12, world, ms)
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: (15.0, 2 * 2.0e12 / 15e-3 / 1e12), 1: (15.0, 2 * 2.0e12 / 15e-3 / 1e12)}


def test_single_process_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)
