"""bench.py's multi-rank aggregation on CPU: two gloo ranks, each a replica
with its own time; the job time is the slowest rank's and the value counts
the bytes of every rank."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    mine = 2.0 if rank == 0 else 5.0              # ms per call on this rank
    ms, value = bench.combine_ranks(mine, 10_000_000, ws, "cpu")
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, ms, value in res:
        assert ms == 5.0
        assert value == pytest.approx(2 * 10_000_000 / 5e-3 / 1e9)


def test_single_rank_is_its_own_time():
    import bench
    ms, value = bench.combine_ranks(4.0, 8_000_000, 1, "cpu")
    assert ms == 4.0 and value == pytest.approx(8_000_000 / 4e-3 / 1e9)
