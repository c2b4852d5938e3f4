"""Multi-process host logic of bench.py on CPU: two gloo ranks, each with its
own seeded batch (replicas, no data-path collective), the job time taken as
the slowest rank's and the throughput summed over ranks."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from segmented_gather_gemv_gb300 import workloads as wl
        # each rank's own batch
        w = wl.decode(seed=bench.replica_seed(rank), M=64, d_in=64, d_out=64)
        ids = torch.from_numpy(w.ids.astype(np.int64))
        gathered = [torch.zeros_like(ids) for _ in range(world)]
        dist.all_gather(gathered, ids)
        # the job time is the slowest rank's
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        out[rank] = (t, all(torch.equal(g, gathered[0]) for g in gathered[1:]))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_and_max_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    times = [out[r][0] for r in range(world)]
    assert times == [15.0, 15.0]              # every rank sees the slowest rank's time
    assert out[0][1] is False                 # the ranks' batches differ (own seed per replica)


def test_whole_job_throughput_sums_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tokens_per_s(1, 100, 256, 2.0)
    two = bench.whole_job_tokens_per_s(2, 100, 256, 2.0)
    assert one == pytest.approx(100 * 256 / 2e-3)
    assert two == pytest.approx(2 * one)
    assert bench.replica_seed(0) != bench.replica_seed(1)
