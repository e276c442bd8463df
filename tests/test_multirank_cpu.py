"""The multi-GPU bench path's host logic, run as two gloo ranks on the CPU.

Every rank runs its own whole problem (replicas: there is no exchange on the data
path); ranks meet only at a barrier and a max-reduction of their timings.  This
checks that machinery with CPU processes, since no GPU test here may use more
than one GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), BENCH_DIST_BACKEND="gloo")
    import bench
    dist, r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(dist, None)
    # each rank reports a different elapsed time; all must agree on the maximum
    slowest = bench.reduce_max(dist, 10.0 + 2.5 * rank)
    bench.barrier(dist, None)
    results[rank] = slowest
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_rank_timing_reduction(world):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {r: 10.0 + 2.5 * (world - 1) for r in range(world)}


def test_aggregate_counts_every_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 3 steps x 1e12 flops in the slowest rank's 2 ms -> 3000 TFLOP/s
    assert bench.aggregate_tflops(2, 1e12, 3, 2.0) == pytest.approx(3000.0)
    assert bench.aggregate_tflops(1, 1e12, 1, 1.0) == pytest.approx(1000.0)


def test_single_process_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    dist, rank, world, local = bench.dist_setup(1)
    assert dist is None and (rank, world, local) == (0, 1, 0)
    assert bench.reduce_max(None, 4.0) == 4.0
