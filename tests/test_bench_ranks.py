"""The replica path of bench.py on CPU: two gloo ranks agree on the slowest
rank's time, the whole-job value counts every rank's bytes, and the
reference arm does no work on ranks other than 0."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.0, 3.5][rank]
        t_max = bench.max_over_ranks(ms)
        out[rank] = (t_max, bench.whole_job_gbs(1e9, world, t_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.5
    # 2 ranks x 1 GB over the slowest rank's 3.5 ms
    assert abs(res[0][1] - 2e9 / 3.5e-3 / 1e9) < 1e-9


def test_single_process_time_unchanged():
    import bench
    assert bench.max_over_ranks(4.25) == 4.25
    assert abs(bench.whole_job_gbs(5e8, 1, 2.0) - 250.0) < 1e-9


def test_reference_arm_idle_on_other_ranks(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1",
                                      "--warmup", "0"])
    assert bench.run_reference(bench.parse()) == 0
    assert capsys.readouterr().out == ""
