"""The cross-rank parts of bench.py (replicas only: one barrier and the max over ranks)
and the reference arm's rank handling, with two gloo ranks on CPU."""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # every rank reports its own step time; the job's is the slowest one's
        ms = bench.max_over_ranks(1.0 + rank, dist, "cpu")
        out.put((rank, ms, bench.job_tokens_per_s(world, 32768, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in res:
        assert ms == 2.0                      # the slower rank's time on every rank
        assert value == pytest.approx(2 * 32768 / 2.0e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_tokens_per_s(1, 1000, 2.0) == pytest.approx(5e5)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=0)
    bench.reference_arm(args, bench.WORKLOADS[bench.DEFAULT_WORKLOAD], 1, 2)
    assert capsys.readouterr().out == ""
