"""Host logic of the multi-replica bench on CPU: two gloo ranks combine their
step times with a max, the whole-job rate counts every replica's work, and the
reference arm runs on rank 0 only."""
import argparse
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports step time 1.5 + r ms and e2e time 10 - r ms
        got = bench.reduce_max_over_ranks([1.5 + rank, 10.0 - rank])
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = dict(q.get(timeout=10) for _ in range(world))
    for r in range(world):
        assert results[r] == [2.5, 10.0]


def test_single_process_reduce_is_identity():
    assert bench.reduce_max_over_ranks([3.0, 4.0]) == [3.0, 4.0]


def test_whole_job_rate_counts_every_replica():
    # 2 replicas x 1e12 flop per step in 2 ms -> 1e15 flop/s
    assert bench.whole_job_rate(1e12, 2.0, 2) == pytest.approx(1e15)
    assert bench.whole_job_rate(5.0, 1.0, 1) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only():
    args = argparse.Namespace(workload="decode_T64", seed=0, steps=2, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None


def test_cast_algorithmic_bytes():
    # one read and two written bytes per scale byte, 4 + 8 bytes per expert
    assert bench.cast_alg_bytes((256, 4096, 128)) == 3 * 256 * 4096 * 128 + 12 * 256
    assert bench.cast_alg_bytes((1, 1, 1)) == 15


def test_cast_reference_arm_runs_on_rank_zero_only():
    args = argparse.Namespace(workload="cast_w13", seed=0, steps=2, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None


def test_cast_oracle_sample_is_bounded():
    # a tiny budget still times at least one expert and reports GB/s > 0
    gbs, ms, sample = bench.run_cast_oracle(1, 1e-6, 0)
    assert gbs > 0 and ms > 0 and "first 1 of 256" in sample


def _failing_worker(rank, world, port, q):
    import datetime
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    if rank == 1:
        # this replica fails between steps and leaves without reducing
        os._exit(3)
    try:
        bench.reduce_max_over_ranks([1.0, 2.0])
        q.put((rank, "returned"))
    except Exception as exc:                     # the peer's exit surfaces as an error
        q.put((rank, type(exc).__name__))


def test_a_replica_that_dies_is_detected_by_the_others():
    """Failure detection on the host: when one replica exits between steps, the
    surviving rank's max-over-ranks reduction ends with an error within the
    process group's timeout instead of hanging."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_failing_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert procs[1].exitcode == 3
    assert procs[0].exitcode == 0
    rank, outcome = q.get(timeout=10)
    assert rank == 0 and outcome != "returned"
