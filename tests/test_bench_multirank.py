"""bench.py's multi-rank logic on CPU: two gloo ranks run as replicas; the job time is
the slowest rank's and the job throughput counts the units of every rank."""
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


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max = bench.max_over_ranks(times[rank], world, "cpu")
        value = bench.job_throughput(1e9, world, ms_max, 1e9)
        out.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    world, times = 2, [10.0, 25.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value in res:
        assert ms_max == 25.0                       # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 1.0 / 0.025)  # 2 ranks x 1 GB in 25 ms = 80 GB/s


def test_single_rank_is_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.job_throughput(5e9, 1, 100.0, 1e9) == pytest.approx(50.0)


def test_reference_arm_prints_only_on_rank_zero(tmp_path, monkeypatch, capsys):
    """Under torchrun the oracle arm runs on rank 0 alone; other ranks exit at once."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    bench.main()
    assert capsys.readouterr().out == ""
