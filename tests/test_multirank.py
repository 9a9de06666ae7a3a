"""The multi-replica path of bench.py on CPU: two gloo ranks.

With --gpus N the bench runs N independent replicas of the decode step (the
path shards by sequence with no exchange); the only cross-rank steps are the
barrier, the slowest rank's time and rank 0's report. These run here as two
gloo processes."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(times[rank], world, "cpu")
        rate = bench.whole_job_rate(1000.0, world, t)
        out_q.put((rank, t, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run_ranks(times):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")  # no fork after the parent imported torch
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, len(times), port, times, q))
          for r in range(len(times))]
    for p in ps:
        p.start()
    got = {}
    for _ in ps:
        rank, t, rate = q.get(timeout=120)
        got[rank] = (t, rate)
    for p in ps:
        p.join(60)
        assert p.exitcode == 0
    return got


def test_two_ranks_agree_on_the_slowest_time_and_the_whole_job_rate():
    got = _run_ranks([0.004, 0.005])  # seconds: rank 1 is the slower one
    for rank in (0, 1):
        t, rate = got[rank]
        assert t == pytest.approx(0.005)
        # both replicas' units over the slowest rank's time
        assert rate == pytest.approx(2 * 1000.0 / 0.005)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25, 1, "cpu") == 0.25
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    args = bench.parse()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""  # the other ranks print nothing
