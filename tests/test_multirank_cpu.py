"""The bench's multi-rank host logic on CPU with two gloo ranks: each rank
runs an independent replica (the operator's batch rows and directions are
independent, so there is no exchange on the data path); the job's time is
the slowest rank's, reduced with one all_reduce(MAX), and its throughput
counts every rank's units."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    ws, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=ws)
    # rank r timed its K steps in (10 + 5r) ms and its end-to-end leg in (30 - r) ms
    total, e2e = bench.max_over_ranks([10.0 + 5 * r, 30.0 - r], dist, "cpu")
    out.put((r, ws, local, total, e2e, bench.job_value(2048, 100, ws, total)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, ws, local, total, e2e, value) in enumerate(res):
        assert (rank, ws, local) == (r, 2, r)
        assert total == 15.0 and e2e == 30.0          # max over the ranks
        assert value == pytest.approx(2048 * 100 * 2 / 0.015)


def test_single_rank_env_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.job_value(2048, 10, 1, 5.0) == pytest.approx(2048 * 10 / 0.005)
