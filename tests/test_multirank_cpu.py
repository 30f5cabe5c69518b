"""The N > 1 path of bench.py on the CPU: two ranks as separate processes on
the gloo backend (one process per GPU on a GPU machine).  Batch-1 decode does not
shard, so N GPUs run N independent replicas with no data-path collective; the
only collectives are the barrier around the timed region and the maximum of
the ranks' times, and the reported value is the units all ranks processed over
the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench

STEPS = 8


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench as b
    w, r, local, pg = b.dist_setup(world)
    ms = 10.0 + 5.0 * r  # the ranks' own timings: rank 1 is the slower one
    pg.barrier()
    slowest = b.max_over_ranks(pg, ms)
    pg.barrier()
    out.put((r, w, local, pg.get_backend(), slowest, b.job_throughput(w, STEPS, slowest / 1e3)))
    pg.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_all_ranks_units():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(out.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for r, (rank, world, local, backend, slowest, value) in enumerate(got):
        assert (rank, world, local, backend) == (r, 2, r, "gloo")
        assert slowest == 15.0  # both ranks see the maximum
        assert value == pytest.approx(2 * STEPS / 0.015)


def test_single_rank_needs_no_collective():
    world, rank, local, pg = bench.dist_setup(1)
    assert (world, rank, local, pg) == (1, 0, 0, None)
    assert bench.max_over_ranks(None, 12.5) == 12.5
    assert bench.job_throughput(1, STEPS, 0.002) == pytest.approx(4000.0)


def test_reference_arm_runs_on_rank_zero_only():
    # rank 1 returns before touching its arguments or the oracle
    assert bench.run_reference(None, 2, 1, None) is None
