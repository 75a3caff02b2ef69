"""The multi-rank timing path of bench.py on CPU: two gloo ranks reduce their
step times to the maximum and compute the same whole-job throughput."""
import os
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = 1.0 + rank            # rank 1 is the slow one
        t = bench.max_over_ranks(step_ms, world)
        out[rank] = (t, bench.job_throughput(1e12, t, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0] == out[1]
    t, value = out[0]
    assert t == 2.0
    assert abs(value - world * 1e12 / 2e-3 / 1e12) < 1e-9   # 1000 TFLOPS


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(2e12, 1.0, 1) == 2000.0
