"""World-size-2 gloo ranks on the CPU: the bench's multi-rank host logic
(rank environment, barrier, max of the step time over ranks, weak-scaling
aggregate).  The data path has no collective, so this is all there is to
test for N > 1 without GPUs."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    step_ms = 1.0 + rank                     # rank 1 is the slow one
    t = bench.max_over_ranks(step_ms, w, "cpu")
    rows_per_rank = 256
    value = rows_per_rank * w / (t * 1e-3)
    q.put((r, local, w, t, value))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, local, world, t, value) in enumerate(res):
        assert rank == r and local == r and world == 2
        assert t == 2.0                      # max over ranks
        assert value == pytest.approx(512 / 2e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    bench.barrier(1)
