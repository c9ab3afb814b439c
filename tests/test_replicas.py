"""The N-GPU bench runs N independent replicas (the path has no exchange step):
the job's timed region is the slowest rank's and the job's throughput is N
replicas' work over it.  Checked on CPU with two gloo ranks."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, dist)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, ms, bench.job_throughput(2e9, ms, world)))


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slower rank's 15 ms; two replicas of 2 GB each in 15 ms
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2] == pytest.approx(2 * 2e9 / 15e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_throughput(1e9, 1000.0, 1) == pytest.approx(1.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(argparse.Namespace(steps=1, warmup=0, gpus=2)) == 0
