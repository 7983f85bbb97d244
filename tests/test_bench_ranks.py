"""The multi-rank path of bench.py on the CPU: two gloo ranks (world size 2).

The hot path shards as independent replicas (each rank runs whole steps on
its own inputs, no data-path collective); the only exchange is the timing
reduction after the timed region, which takes the slowest rank's step time.
Checked here: that reduction returns the element-wise maximum on every rank,
the whole-job throughput scales with the number of replicas at equal step
time, and the reference arm does no work on ranks other than 0."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        # rank 0 is slower on the first value, rank 1 on the second
        mine = [10.0 + 5.0 * (rank == 0), 3.0 + 4.0 * (rank == 1)]
        got = bench.max_over_ranks(mine)
        dist.barrier()
        q.put((rank, got, None))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, None, repr(e)))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in procs:
            rank, got, err = q.get(timeout=120)
            assert err is None, f"rank {rank}: {err}"
            results[rank] = got
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert results == {0: [15.0, 7.0], 1: [15.0, 7.0]}
    assert all(p.exitcode == 0 for p in procs)


def test_single_process_values_pass_through():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def test_whole_job_throughput_counts_every_replica():
    import bench
    one = bench.whole_job_tflops(0.2, 1)
    assert bench.whole_job_tflops(0.2, 2) == pytest.approx(2 * one)
    assert bench.whole_job_tflops(0.4, 2) == pytest.approx(one)
    # 3 GEMMs of 2*4096^3 FLOPs each in 0.2 ms
    assert one == pytest.approx(3 * 2 * 4096 ** 3 / 0.2e-3 / 1e12)


def test_reference_arm_other_ranks_do_nothing():
    import bench
    assert bench.reference_arm(None, 1, 2) is None
