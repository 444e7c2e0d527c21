"""The N > 1 bench path, on CPU: independent replicas (no data-path
collective), timed by the slowest rank.  Two gloo ranks on 127.0.0.1 check
the max-over-ranks reduction and the whole-job throughput; the reference arm
runs on rank 0 only."""

import argparse
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench as b
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = b.dist_env()
        # each rank's "median timed region": the job is as slow as its slowest rank
        region_ms = b.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        q.put((r, w, lr, region_ms, b.job_throughput(w, 1e9, region_ms / 100)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        out = sorted(q.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert [(r, w, lr) for r, w, lr, _, _ in out] == [(0, 2, 0), (1, 2, 1)]
    assert all(ms == 15.0 for _, _, _, ms, _ in out)                 # max over ranks
    # 2 replicas x 1 GB per step in 0.15 ms per step
    assert all(v == pytest.approx(2 * 1e9 / 0.15e-3 / 1e12) for *_, v in out)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_throughput(1, 5e11, 1000.0) == pytest.approx(0.5)
    assert bench.job_throughput(4, 5e11, 1000.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = argparse.Namespace(workload="small", steps=1, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None
    assert capsys.readouterr().out == ""
