"""The multi-rank path of the benchmark on CPU: two gloo ranks (no GPU).

Rows are independent, so every rank convolves its own replica of the
workload with no collective on the data path; the only cross-rank steps are
the barrier and the maximum of the step times, which these tests run."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import workloads as W
    r, wsz, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=wsz)
    ms = 1.5 + rank  # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, wsz, torch.device("cpu"))
    dist.barrier()
    w = W.scaled(W.WORKLOADS["causal-1k"], B=1, H=2, N=1024)
    u = W.make_inputs(w, seed=r)["u"].f64  # the replica of this rank (seed = rank)
    q.put((r, wsz, local, slowest, bench.job_value(w.outputs, wsz, slowest), float(u.sum())))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_job_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 and r[2] == r[0] for r in res)
    assert all(r[3] == 2.5 for r in res)  # max over ranks, seen by every rank
    outputs = 1 * 2 * 1024
    assert all(abs(r[4] - 2 * outputs / 2.5e-3) < 1e-6 * r[4] for r in res)  # both replicas over the slowest time
    assert res[0][5] != res[1][5]  # distinct seeded replicas per rank


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1, None) == 3.0
    assert bench.job_value(1000, 1, 2.0) == 1000 / 2e-3
