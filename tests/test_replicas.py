"""The multi-GPU form of the bench: independent replicas (the layer has no exchange step).
Checked here with two gloo ranks on the CPU: every rank sees the slowest rank's time, the
job's throughput counts all ranks' tokens over that time, and the reference arm runs on rank
0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + 5.0 * rank, 3.0 - rank]  # rank 1 is slower on the first timing
        got = bench.max_over_ranks(mine)
        ws, r, local = bench.dist_env()
        q.put((rank, got, (ws, r, local)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_env_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, env in res:
        assert got == [15.0, 3.0]
        assert env == (2, rank, rank)


def test_replica_throughput_counts_all_ranks():
    import bench
    assert bench.replica_throughput(1, 10, 128, 20.0) == pytest.approx(64000.0)
    # two replicas of 10 steps x 128 tokens; the slower takes 25 ms in all
    assert bench.replica_throughput(2, 10, 128, 25.0) == pytest.approx(102400.0)
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]  # no process group: identity


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "workload_data", lambda *a, **k: called.append(1))
    args = type("A", (), {"workload": "dsv3_T128", "steps": 1, "warmup": 3})()
    assert bench.run_reference(args) is None
    assert not called
