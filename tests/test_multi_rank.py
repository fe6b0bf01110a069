"""Host logic of bench.py's multi-GPU path (replicas, one rank per GPU) on
world-size-2 gloo process groups on the CPU: the environment it reads, the
max-over-ranks timing reduction and the whole-job rate, and the reference arm
running on rank 0 only."""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w, r, l = bench.dist_setup()
        # rank 0 is slower on the first timing, rank 1 on the second
        got = bench.max_over_ranks(w, [10.0 + 5.0 * (rank == 0), 7.0 + 2.0 * (rank == 1)], "cpu")
        rate = bench.whole_job_rate(w, 16384, 4, got[0])
        q.put((rank, w, r, l, got, rate))
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, rr, l, got, rate) in enumerate(res):
        assert (r, w, rr, l) == (rank, 2, rank, rank)
        assert got == [15.0, 9.0]          # max over the two ranks, per value
        assert rate == pytest.approx(2 * 16384 * 4 / 15e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1, [3.5, 2], "cpu") == [3.5, 2.0]
    assert bench.whole_job_rate(1, 1000, 2, 4.0) == pytest.approx(5e5)


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    called = []
    monkeypatch.setattr(bench, "cpu_baseline_oracle", lambda *a, **k: called.append(a))
    bench.run_reference(argparse.Namespace(steps=2, warmup=1))
    assert called == [] and capsys.readouterr().out == ""
