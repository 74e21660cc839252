"""The N > 1 host logic of bench.py on CPU: two gloo ranks, as torchrun would
start them.  The decode step has no exchange (every (request, KV head) unit is
independent), so the only cross-rank steps are the barrier and the max of the
per-rank times; the job's throughput counts every rank's replica."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w = bench.dist_init(None)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    t = 0.5 + rank  # rank 1 is the slow one
    t_max = bench.max_over_ranks(t, w)
    q.put((rank, t_max, bench.job_throughput(32, 10, t_max, w)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t_max, value in got:
        assert t_max == 1.5
        assert value == 2 * 32 * 10 / 1.5


def test_single_rank_is_plain_throughput():
    assert bench.max_over_ranks(2.0, 1) == 2.0
    assert bench.job_throughput(32, 20, 0.5, 1) == 32 * 20 / 0.5
