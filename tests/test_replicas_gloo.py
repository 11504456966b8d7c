"""The multi-GPU form of the bench: independent replicas, max over ranks.

The layer is data-parallel over tokens with replicated weights and has no
exchange step, so N GPUs run N replicas. What the ranks share is host logic:
a barrier around the timed region and the max over ranks of the measured step
times. This runs that logic on two CPU processes over gloo.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    r = bench.Ranks(rank, world, rank, backend="gloo")
    try:
        r.barrier()
        # rank 1 is slower on the device time, rank 0 on the end-to-end time
        ms, e2e = r.max([0.5 + 0.25 * rank, 2.0 - 0.5 * rank])
        out.put((rank, ms, e2e, bench.throughput(16, world, ms)))
        r.barrier()
    finally:
        r.close()


@pytest.mark.timeout(120)
def test_two_replicas_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=90) for _ in range(world))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, ms, e2e, value in got:
        assert ms == 0.75 and e2e == 2.0
        # whole job: 2 replicas x 16 tokens in the slowest rank's 0.75 ms
        assert value == pytest.approx(2 * 16 / 0.75e-3)


def test_single_rank_needs_no_process_group():
    r = bench.Ranks(0, 1, 0)
    r.barrier()
    assert r.max([1, 2.5]) == [1.0, 2.5]
    r.close()
    assert bench.throughput(4096, 1, 2.0) == pytest.approx(2048000.0)


def test_reference_arm_runs_on_rank_zero_only():
    import argparse
    args = argparse.Namespace(config=1, steps=1, warmup=3)
    assert bench.run_reference(args, 1, 2) is None
