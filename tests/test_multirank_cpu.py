"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

With N GPUs every rank runs its own replica of the workload; the only
collectives are the barrier and the max-over-ranks of the timed region, and
the job's value is the units all ranks processed over the slowest rank's time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    elapsed = 1.0 + 0.5 * r          # rank 1 is the slow one
    slowest = bench.max_over_ranks(dist, elapsed)
    value = bench.job_value(1000.0, w, slowest)
    bench.barrier(dist)
    dist.destroy_process_group()
    q.put((r, local, slowest, value))


def test_two_rank_timing_is_max_and_value_is_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, local, slowest, value in res:
        assert slowest == pytest.approx(1.5)
        assert value == pytest.approx(2 * 1000.0 / 1.5)
    assert [x[0] for x in res] == [0, 1]


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.parse_args(["--impl", "reference"])) is None
