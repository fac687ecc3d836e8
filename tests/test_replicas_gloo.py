"""Replica (data-parallel) host logic of bench.py on two CPU ranks over gloo.

The path shards into independent row chunks, so N GPUs run N replicas with no data-path
collective; the only cross-rank step is the max over ranks of the timed region, from which the
whole-job throughput is computed.  This runs two real processes with a gloo process group.
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


def _rank_main(rank, world, port, times, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(times[rank], "cpu")
        v = bench.replica_throughput(world, 256, 20, t)
        q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [3.5, 4.25]  # ms of the timed region on each rank
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time, and report the same whole-job value
    assert [r[1] for r in res] == [4.25, 4.25]
    assert res[0][2] == res[1][2] == pytest.approx(2 * 256 * 20 / 4.25e-3)


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(2.5, "cpu") == 2.5
    assert bench.replica_throughput(1, 256, 20, 2.0) == pytest.approx(256 * 20 / 2e-3)
