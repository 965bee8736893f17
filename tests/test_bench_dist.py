"""The benchmark's multi-rank logic on CPU: two gloo ranks (127.0.0.1), the
barrier, the max-over-ranks timing, the whole-job rate, and the reference arm
running on rank 0 only."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w)
    bench.barrier(dist)
    slowest = bench.max_over_ranks(dist, 10.0 + 5.0 * r)     # rank 1 is the slow one
    rate = bench.job_rate(2_000_000_000, w, 4, slowest)
    bench.barrier(dist)
    dist.destroy_process_group()
    out.put((r, slowest, rate))


def test_two_gloo_ranks_agree_on_slowest_time_and_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in results] == [0, 1]
    for _, slowest, rate in results:
        assert slowest == 15.0
        # 2 ranks x 4 steps x 2 GFLOP in 15 ms.
        assert rate == pytest.approx(2 * 4 * 2.0 / 15e-3)


def test_job_rate_single_rank():
    assert bench.job_rate(355_409_000_000, 1, 50, 380.0) == pytest.approx(46764.3, rel=1e-4)


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        workload, steps, warmup, ref_step_seconds = "c1", 1, 0, 0.01
    assert bench.run_reference(Args(), 2, 1) is None
    line = bench.run_reference(Args(), 1, 0)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
