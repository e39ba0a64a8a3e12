"""Multi-rank bench logic on CPU (gloo, world size 2): every rank runs an
independent replica; the job time is the slowest rank's and the throughput
sums the ranks' work. The layer itself needs no collective."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [3.0, 5.0][rank]
    worst = bench.max_over_ranks(ms, "cpu", world)
    out[rank] = (worst, bench.job_throughput(1000.0, world, worst))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_max_time_and_summed_work():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    worst, thr = out[0]
    assert worst == 5.0
    assert thr == pytest.approx(2 * 1000.0 / 5e-3)


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(2.5, "cpu", 1) == 2.5
    assert bench.job_throughput(10.0, 1, 2.0) == pytest.approx(5000.0)
