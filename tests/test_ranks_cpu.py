"""The multi-replica path of bench.py on CPU: two gloo ranks (world size 2).

With --gpus N > 1 every rank runs an independent replica of the block; the ranks
meet only at the barriers around the timed region and in the maximum over their
step times, and the job's throughput is all replicas' FLOPs over the slowest
replica's time.  These tests run that host logic with two processes on the
CPU, and check that the reference arm does its work on rank 0 only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, step_ms, flops, q):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        bench.rank_barrier(world)
        ms_max = bench.max_over_ranks(step_ms[rank], world)
        value = bench.job_throughput(flops, world, ms_max)
        bench.rank_barrier(world)
        q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_replica():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    step_ms = [4.8, 5.1]  # rank 1 is the slower replica
    flops = 7.422e12
    procs = [ctx.Process(target=_worker, args=(r, 2, port, step_ms, flops, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, ms_max, value in results:
        assert ms_max == pytest.approx(5.1)
        assert value == pytest.approx(2 * flops / 5.1e-3 / 1e12)


def test_one_rank_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_throughput(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    """Under torchrun the other ranks of --impl reference exit 0 without work."""
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""
