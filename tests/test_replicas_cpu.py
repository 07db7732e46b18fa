"""The N > 1 bench path ("replicas only": every rank runs the whole
workload, no data-path collective) on CPU ranks with gloo: the job's time is
the slowest rank's, its throughput counts every rank's work; the reference
arm runs on rank 0 only."""
import os
import socket
import types

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, value = bench.job_throughput(10.0 * (rank + 1), 3.0e12, world, dist, "cpu")
        q.put((rank, ms, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_take_the_slowest_rank(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.start_processes(_rank_main, args=(world, _free_port(), q), nprocs=world,
                       start_method="spawn", join=True)
    got = sorted(q.get(timeout=60) for _ in range(world))
    assert [r for r, _, _ in got] == list(range(world))
    slowest = 10.0 * world
    for _, ms, value in got:
        assert ms == slowest                      # max over ranks, on every rank
        assert value == pytest.approx(3.0e12 * world / (slowest * 1e-3) / 1e12)


def test_single_rank_needs_no_collective():
    ms, value = bench.job_throughput(4.0, 2.0e12, 1)
    assert ms == 4.0 and value == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = types.SimpleNamespace(workload="fp8_linear_add", steps=1, warmup=3, ref_rows=1)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
