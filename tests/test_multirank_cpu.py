"""The benchmark's N>1 host logic on CPU: two gloo ranks.

Each (b, h) head is independent, so ranks run independent batches (weak
scaling) and exchange only one timing scalar: the whole-job throughput is the
units of all ranks over the slowest rank's time.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    t_ms = [2.0, 5.0][rank]                     # rank 1 is the slow one
    value, t = bench.aggregate(10.0, t_ms, world)
    q.put((rank, value, t))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, t in got:
        assert t == 5.0
        assert value == pytest.approx(10.0 * 2 / 5e-3)


def test_single_rank_is_identity():
    import bench
    value, t = bench.aggregate(10.0, 4.0, 1)
    assert t == 4.0 and value == pytest.approx(10.0 / 4e-3)
