"""The multi-rank host logic of bench.py on world_size-2 gloo ranks (CPU).

bench.py runs one replica of the workload per GPU; the ranks share only a
barrier around the timed region and the max over ranks of its duration.
Here two CPU processes exercise exactly those calls.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    n, r, local = bench.dist_setup(backend="gloo")
    assert (n, r, local) == (ws, rank, rank)
    bench.barrier(n)
    # each rank's timed duration differs; the job's is the slowest
    t = bench.max_over_ranks(10.0 + 5.0 * rank, n)
    v = bench.job_throughput(256, t, n)
    out.put((rank, t, v))
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_over_ranks():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(ws))
    for rank, t, v in got:
        assert t == 15.0                       # max over ranks, identical on every rank
        assert v == pytest.approx(256 * 2 / 15.0)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(100, 2.0, 1) == 50.0
