"""Instance sharding and the search's final reduction across ranks, exercised
with two gloo ranks on the CPU (one process per rank)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from pipeline_schedule_simulation_gb300.sharding import best_of, shard_range


def test_shard_range_covers_exactly():
    for n in (0, 1, 7, 65536, 1000003):
        for world in (1, 2, 3, 8):
            got = [shard_range(n, r, world) for r in range(world)]
            assert got[0][0] == 0 and got[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(got, got[1:]))
            sizes = [hi - lo for lo, hi in got]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_range(5, 2, 2)


def test_best_of_ties_and_infeasible():
    assert best_of([(10, 5), (10, 3), (11, 0)]) == (10, 3)
    assert best_of([(-1, -1), (-1, -1)]) == (-1, -1)
    assert best_of([(-1, -1), (7, 9)]) == (7, 9)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    from pipeline_schedule_simulation_gb300.sharding import reduce_best, shard_range
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lo, hi = shard_range(101, rank, world)
    # each rank's local best over a made-up score table with a tie across ranks
    scores = {i: (i * 37) % 11 + 5 for i in range(101)}
    scores[13] = scores[77] = 1
    local = min((scores[i], i) for i in range(lo, hi))
    results[rank] = reduce_best(*local)
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_best_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert results[0] == results[1] == (1, 13)
