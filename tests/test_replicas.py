"""The multi-GPU path of the benchmark is replicas only: the ranks share no data, meet at a
barrier around the timed region, and the job's time is the max over ranks. This checks that
host-side glue with two gloo ranks on the CPU (no GPU)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    bench.init_dist(w, local, backend="gloo")
    bench.barrier(w)
    t = bench.allreduce_max(10.0 + 5.0 * r, w)  # each replica reports its own time
    bench.barrier(w)
    bench.close_dist()
    q.put((r, w, t))


@pytest.mark.timeout(120)
def test_two_replicas_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert got == [(0, 2, 15.0), (1, 2, 15.0)]


def test_single_process_needs_no_group():
    import bench
    assert bench.allreduce_max(3.5, 1) == 3.5
    bench.barrier(1)
