"""The multi-rank bench logic on CPU: two gloo ranks, independent replicas.

The layer has no exchange step, so N GPUs run N replicas; the job time is the
slowest rank's and the throughput counts every rank's work.  This checks that
aggregation with a real two-process gloo group (no GPU involved).
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                 # rank 1 is the slow one
        slowest = bench.max_over_ranks(mine)
        tflops = bench.job_tflops(2e12, steps=4, world=world, max_total_ms=slowest)
        out.put((rank, slowest, tflops))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_count_all_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for _, slowest, tflops in got:
        assert slowest == pytest.approx(15.0)
        # 2 ranks x 4 steps x 2e12 flop in 15 ms
        assert tflops == pytest.approx(2 * 4 * 2e12 / 15e-3 / 1e12)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1e12, 10, 1, 10.0) == pytest.approx(1000.0)
