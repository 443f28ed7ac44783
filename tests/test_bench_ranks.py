"""The multi-GPU bench path on CPU: two gloo ranks agree on the slowest
rank's time and on the whole-job rate (independent replicas, weak scaling)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    r, local, w = bench.dist_setup("gloo")
    assert (r, local, w) == (rank, rank, world)
    ms = 100.0 + 50.0 * rank            # rank 1 is the slowest
    bench.barrier(w)
    m = bench.reduce_max(ms, w)
    out[rank] = (m, bench.whole_job_rate(10, w, m))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    m, rate = out[0]
    assert m == 150.0
    assert rate == pytest.approx(10 * 2 / 0.150)


def test_single_rank_rate():
    assert bench.reduce_max(12.5, 1) == 12.5
    assert bench.whole_job_rate(100, 1, 50.0) == pytest.approx(2000.0)
