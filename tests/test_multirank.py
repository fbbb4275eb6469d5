"""The benchmark's multi-rank harness on CPU: two gloo ranks, 127.0.0.1.

Each rank runs an independent replica of the workload; the only cross-rank
traffic is the barrier and the max-over-ranks of the timed interval.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench

    env = bench.dist_env()
    t = bench.max_over_ranks(0.5 + rank, ws, device="cpu")  # slowest rank's time wins
    bench.barrier(ws)
    q.put((rank, env, t))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got = {rank: (env, t) for rank, env, t in out}
    for rank in (0, 1):
        env, t = got[rank]
        assert env == (2, rank, rank)
        assert t == pytest.approx(1.5)


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
