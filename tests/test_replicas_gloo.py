"""The benchmark's multi-rank bookkeeping (replicas, no data exchange): two
gloo ranks on the CPU agree on the job time (the slowest rank's) and on the
per-row figure computed from the rows all ranks processed."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    d = bench.init_dist(w, "gloo")
    bench.barrier(d)
    my_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    job_ms = bench.max_over_ranks(d, my_ms)
    steps, batch = 100, 1
    us_per_row = job_ms * 1e3 / (steps * batch * w)
    q.put((rank, w, r, job_ms, us_per_row))
    d.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 and r[2] == r[0] for r in res)
    assert all(r[3] == 15.0 for r in res)
    assert all(abs(r[4] - 15.0 * 1e3 / 200) < 1e-9 for r in res)


def test_single_process_needs_no_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
