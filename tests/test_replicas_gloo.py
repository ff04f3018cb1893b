"""The multi-rank (replicas) path of bench.py on CPU: world size 2 over gloo.

On GPUs each rank runs an independent replica of the GEMM (no exchange on the
data path); the only cross-rank steps are the max-over-ranks timing and the
whole-job value.  Those are checked here with CPU tensors."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(1.0 + rank, world, torch.device("cpu"))  # rank 1 is the slower one
        q.put((rank, ms, bench.job_tflops(2.0e12, world, ms)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time_and_value():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    for rank, ms, value in got:
        assert ms == 2.0                      # max over ranks, on every rank
        assert value == pytest.approx(2000.0)  # 2 ranks x 2e12 FLOP / 2 ms = 2000 TFLOP/s


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(3.5, 1, None) == 3.5


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 3, 3
    assert bench.run_reference(Args()) == 0
