"""The bench's multi-rank path on the CPU: two gloo ranks on 127.0.0.1 (the
path runs replicas and shares only the slowest rank's time), and the
reference arm printing on rank 0 only."""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
    dist.barrier()
    ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
    out[rank] = (ms, bench.replica_rate(1000, world, 3, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == out[1]
    ms, rate = out[0]
    assert ms == 20.0
    assert rate == pytest.approx(1000 * world * 3 / 0.020)


def test_single_process_passes_time_through():
    assert bench.max_over_ranks(12.5, None, None) == 12.5
    assert bench.replica_rate(10, 1, 2, 1000.0) == pytest.approx(20.0)


def test_reference_arm_is_silent_off_rank_zero(capsys):
    class A:
        workload = "homogeneous"
        warmup = 0
        steps = 1
        ref_budget = 0.1
    bench.run_reference(A(), rank=1, world=2)
    assert capsys.readouterr().out == ""
