"""World-size-2 checks of bench.py's multi-rank plumbing on CPU (gloo).

Requests are independent, so ranks share no data: each rank runs its own
batch from its own seed, and only the timing is combined (barrier, max of the
per-rank times, sum of the units).  These tests run that combination and the
reference arm's rank rule with two gloo processes.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, n, local = bench.dist_setup()
    assert (r, n, local) == (rank, ws, rank)
    assert dist.get_backend() == "gloo"
    # rank r processed 1000·(r+1) units in 10·(r+1) ms: the job rate divides
    # all units by the slowest rank's time
    value, ms = bench.job_throughput(1000.0 * (rank + 1), 10.0 * (rank + 1), ws)
    bench.barrier(ws)
    # the reference arm: rank 0 alone works and prints, the others return at once
    printed = None
    if rank != 0:
        class Args:
            steps, warmup, gpus = 1, 0, ws
        printed = bench.run_reference(Args(), rank, ws)
    seed = bench.SEED + 7919 * rank
    dist.destroy_process_group()
    q.put((rank, value, ms, printed, seed))


def test_two_rank_job_throughput_and_reference_rank_rule():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, value, ms, printed, seed = q.get(timeout=120)
        res[rank] = (value, ms, printed, seed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        value, ms, _, _ = res[rank]
        assert ms == pytest.approx(20.0)
        assert value == pytest.approx(3000.0 / 0.020)
    assert res[1][2] is None
    assert res[0][3] != res[1][3]            # every rank draws its own requests


def test_single_rank_job_throughput():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.job_throughput(500.0, 250.0, 1)
    assert ms == 250.0 and value == pytest.approx(2000.0)
