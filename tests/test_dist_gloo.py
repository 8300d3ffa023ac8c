"""The multi-rank host path on CPU with the gloo backend (world size 2):
shares cover every unit once, replicas get distinct seeds, and the timing
reduction takes the slowest rank and the summed work."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from transformer_head_scaled_sdpa_gb300 import dist as mdist


def test_shard_covers_every_unit_once():
    for total in (0, 1, 7, 64, 1000):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                a, b = mdist.shard(total, r, world)
                assert 0 <= a <= b <= total
                seen.extend(range(a, b))
            assert seen == list(range(total))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w = mdist.init("gloo")
    assert (r, w) == (rank, world)
    mdist.barrier()
    elapsed = 1.0 + rank           # rank 1 is the slow one
    units = 100 * (rank + 1)
    t = mdist.max_over_ranks(elapsed)
    u = mdist.sum_over_ranks(units)
    q.put((rank, t, u, mdist.rank_seed(1004, rank)))
    mdist.finish()


@pytest.mark.timeout(120)
def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [x[1] for x in res] == [2.0, 2.0]
    assert [x[2] for x in res] == [300.0, 300.0]
    assert res[0][3] != res[1][3]
