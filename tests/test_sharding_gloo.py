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


def _shard_worker(rank, world, port, results):
    """One rank: its instance range of a real batch and its candidate range of
    the 80-layer search, scored by the CPU oracle (the rank's GPU call on a
    box with GPUs), then the same exchange the benchmark's ranks do."""
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    import pipeline_schedule_simulation_gb300.workloads as W
    from pipeline_schedule_simulation_gb300.sharding import reduce_best, shard_range
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # evaluation: instances [lo, hi) of a heterogeneous 1F1B batch
    b = W.hetero_1f1b(n=1001, seed=12)
    lo, hi = shard_range(b.n, rank, world)
    m = hi - lo
    cf = b.cost_f.reshape(b.P, b.M, b.n)[:, :, lo:hi].copy().reshape(-1)
    cb = b.cost_b.reshape(b.P, b.M, b.n)[:, :, lo:hi].copy().reshape(-1)
    cm = b.comm.reshape(b.P - 1, b.n)[:, lo:hi].copy().reshape(-1)
    r = oracle.eval_batch(b.policy, b.P, b.M, 1, cf, cb, (1, b.M * m, m), comm=cm, comm_strides=(1, m), n=m)
    width = -(-b.n // world)
    mine = torch.full((width,), -1, dtype=torch.int64)
    mine[:m] = torch.from_numpy(r["makespan"].astype(np.int64))
    got = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(got, mine)
    sizes = [shard_range(b.n, q, world) for q in range(world)]
    results[f"eval{rank}"] = np.concatenate([got[q][:hi_ - lo_].numpy() for q, (lo_, hi_) in enumerate(sizes)])
    # search: candidates [lo, hi) of the 80-layer problem, then the global best
    p = W.layer_split(n_cand=3000)
    lo, hi = shard_range(p.n_cand, rank, world)
    s = oracle.search(p.layer_tf, p.layer_tb, p.layer_act, p.P, p.M, p.comm, p.cap, p.seed, lo, hi)
    results[f"search{rank}"] = reduce_best(s["best_makespan"], s["best_idx"])
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_evaluation_and_search_two_gloo_ranks(orc):
    """Two ranks split a real batch and a real candidate range with
    shard_range: the gathered makespans equal the whole batch's, and
    reduce_best returns the whole range's winner (ties to the lower index)."""
    import numpy as np

    import pipeline_schedule_simulation_gb300.workloads as W
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    b = W.hetero_1f1b(n=1001, seed=12)
    whole = orc.eval_batch(b.policy, b.P, b.M, 1, b.cost_f, b.cost_b, b.strides, comm=b.comm,
                           comm_strides=b.comm_strides, n=b.n)
    for rank in (0, 1):
        assert np.array_equal(results[f"eval{rank}"], whole["makespan"])
    p = W.layer_split(n_cand=3000)
    s = orc.search(p.layer_tf, p.layer_tb, p.layer_act, p.P, p.M, p.comm, p.cap, p.seed, 0, p.n_cand)
    assert s["best_idx"] >= 0
    assert results["search0"] == results["search1"] == (s["best_makespan"], s["best_idx"])
