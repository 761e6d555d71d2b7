"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks (replicas of the decode
step, one per GPU on a real node) agree on the job time (the slowest rank's), the
whole-job rate counts every rank's units, and every rank draws its own inputs."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        job_ms = bench.max_over_ranks(ms, dist, "cpu")
        dist.barrier()
        out[rank] = (job_ms, bench.job_rate(4, world, job_ms), bench.rank_seed(1005, rank))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_job_time_and_rate():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == res[1][1] == 4 * 2 / 15e-3
    assert res[0][2] != res[1][2]


def test_single_rank_is_its_own_job():
    assert bench.max_over_ranks(7.5, None, "cpu") == 7.5
    assert bench.job_rate(4, 1, 100.0) == 40.0
    assert bench.rank_seed(1005, 0) == 1005
