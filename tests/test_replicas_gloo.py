"""The multi-GPU path of the benchmark is replicas only: independent ranks,
one barrier and a max over the ranks' times, whole-job throughput over the
slowest rank. Its host logic runs here as two gloo ranks on the CPU."""
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


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.5, 4.0][rank]                    # the second replica is slower
        dist.barrier()
        m = bench.replica_max(ms, world, "cpu")
        v = bench.replica_value(1e9, world, m)   # 1 GB per replica
        out.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 4.0                          # both ranks see the max
        assert v == pytest.approx(2 * 1e9 / 4e-3 / 1e9)  # 2 GB over 4 ms = 500 GB/s


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_max(3.0, 1, "cpu") == 3.0
    assert bench.replica_value(2e9, 1, 4.0) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun the oracle arm runs and prints on rank 0 only; the other
    ranks return at once, without touching the oracle."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup, workload = 1, 0, bench.DEFAULT_WORKLOAD
    assert bench.run_reference(Args()) is None
