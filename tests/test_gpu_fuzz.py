"""Seeded random shapes for every evaluator and search, against the oracle.

The hand-picked shapes of the other parity tests cover the limits and the
kernels' switch points; these cases draw P, M, v, the policy, the layout
(instance-minor with a random row padding, or instance-major), the batch size
and the cost ranges at random (fixed seeds), so that combinations nobody
picked are checked too.  Costs include zeros where the schedule allows them
(GPipe, 1F1B and interleaved; Zero Bubble and DualPipe need F and B >= 1)."""
import os

import numpy as np
import pytest

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import (assert_same, assert_same_zb, run_gpu, run_gpu_dp, run_gpu_zb, run_oracle, run_oracle_dp,
                         run_oracle_zb)

pytestmark = pytest.mark.gpu

NCPU = os.cpu_count() or 8


def _shape(rng):
    policy = int(rng.choice([W.GPIPE, W.ONEF1B, W.INTERLEAVED, W.GPIPE_FIFO]))
    P = int(rng.integers(1, 17))
    if policy == W.INTERLEAVED:
        v = int(rng.integers(2, max(3, min(8, 64 // P) + 1)))
        M = P * int(rng.integers(1, 5))
    else:
        v = 1
        M = int(rng.integers(1, 41))
    return policy, P, M, v


@pytest.mark.parametrize("seed", range(24))
def test_eval_random_shapes(orc, seed):
    rng = np.random.default_rng(1000 + seed)
    for _ in range(16):
        policy, P, M, v = _shape(rng)
        n = int(rng.integers(1, 140))
        layout = "inst_minor" if rng.random() < 0.6 else "inst_major"
        hi = int(rng.choice([3, 20, 500]))
        b = W.random_batch(policy, P, M, v, n, seed=int(rng.integers(1 << 30)), lo=0, hi=hi,
                           comm_hi=int(rng.integers(0, 7)), layout=layout, pad_to=int(rng.choice([1, 4, 8])),
                           stride_mb_zero=bool(rng.random() < 0.25))
        g = run_gpu(b, op_times=True)
        r = run_oracle(orc, b, op_times=True, nthreads=NCPU)
        assert_same(g, r, op_times=True)


@pytest.mark.parametrize("seed", range(8))
def test_zero_bubble_random_shapes(orc, seed):
    rng = np.random.default_rng(2000 + seed)
    for _ in range(16):
        policy = int(rng.choice([W.ZB1P, W.ZB2P]))
        P, M = int(rng.integers(1, 17)), int(rng.integers(1, 41))
        n = int(rng.integers(1, 140))
        b = W.random_zb(policy, P, M, n, seed=int(rng.integers(1 << 30)), lo=1, hi=int(rng.choice([3, 20, 300])),
                        w_lo=0, w_hi=int(rng.choice([0, 5, 300])), comm_hi=int(rng.integers(0, 7)),
                        layout="inst_minor" if rng.random() < 0.5 else "inst_major",
                        pad_to=int(rng.choice([1, 4])))
        g = run_gpu_zb(b, op_times=True)
        r = run_oracle_zb(orc, b, op_times=True, nthreads=NCPU)
        assert_same_zb(g, r, op_times=True)


@pytest.mark.parametrize("seed", range(8))
def test_dualpipe_random_shapes(orc, seed):
    rng = np.random.default_rng(3000 + seed)
    for _ in range(16):
        P, M = int(rng.integers(1, 17)), int(rng.integers(1, 41))
        m_a = int(rng.integers(0, M + 1))
        n = int(rng.integers(1, 140))
        b = W.random_batch(W.ONEF1B, P, M, 1, n, seed=int(rng.integers(1 << 30)), lo=1,
                           hi=int(rng.choice([3, 20, 300])), comm_hi=int(rng.integers(0, 7)),
                           layout="inst_minor" if rng.random() < 0.5 else "inst_major",
                           stride_mb_zero=bool(rng.random() < 0.2))
        g = run_gpu_dp(b, m_a, op_times=True)
        r = run_oracle_dp(orc, b, m_a, op_times=True, nthreads=NCPU)
        assert_same_zb(g, r, op_times=True)


def _layers(rng, L):
    return (rng.integers(1, int(rng.choice([5, 40, 200])), L).astype(np.int32),
            rng.integers(1, int(rng.choice([5, 80, 400])), L).astype(np.int32),
            rng.integers(1, int(rng.choice([3, 50])), L).astype(np.int64))


def _check_search(got, ref, ncut):
    import torch
    torch.cuda.synchronize()
    assert np.array_equal(got["all_makespan"].cpu().numpy(), ref["all_makespan"])
    assert int(got["best_idx"].item()) == ref["best_idx"]
    assert int(got["best_makespan"].item()) == ref["best_makespan"]
    if ref["best_idx"] >= 0:
        # the buffer holds at least one word; a one-stage split has no cuts
        assert list(got["best_cuts"].cpu().numpy()[:ncut]) == list(ref["first"][1:ncut + 1])


@pytest.mark.parametrize("seed", range(6))
def test_searches_random_problems(orc, seed):
    """The seeded, exhaustive and interleaved searches on random problems:
    every candidate's makespan (or rejection), the winner and its cuts."""
    from gpu_helpers import to_dev
    from pipeline_schedule_simulation_gb300 import binding as B
    rng = np.random.default_rng(4000 + seed)
    for _ in range(4):
        P = int(rng.integers(1, 9))
        L = int(rng.integers(P, 3 * P + 12))
        M = int(rng.integers(1, 40))
        comm = int(rng.integers(0, 5))
        ltf, ltb, lact = _layers(rng, L)
        cap = int(lact.sum() * rng.choice([0.3, 1.0, 10.0])) * max(1, min(P, M))
        d = [to_dev(x) for x in (ltf, ltb, lact)]
        sd = int(rng.integers(1 << 40))
        c0, n = int(rng.integers(0, 50)), int(rng.integers(1, 700))
        _check_search(B.partition_search(*d, P, M, comm, cap, sd, c0, n, all_makespan=True),
                      orc.search(ltf, ltb, lact, P, M, comm, cap, sd, c0, c0 + n, nthreads=NCPU), P - 1)
        total = int(orc.binom(L - 1, P - 1))
        r0 = int(rng.integers(0, total))
        nr = min(600, total - r0)
        _check_search(B.partition_search_ranks(*d, P, M, comm, cap, r0, nr, all_makespan=True),
                      orc.search_ranks(ltf, ltb, lact, P, M, comm, cap, r0, r0 + nr, nthreads=NCPU), P - 1)
        # interleaved: v >= 2 chunks per device, M a multiple of P, L >= P*v layers
        Pi = int(rng.integers(1, 5))
        v = int(rng.integers(2, 4))
        Li = int(rng.integers(Pi * v, Pi * v + 10))
        Mi = Pi * int(rng.integers(1, 5))
        ltf, ltb, lact = _layers(rng, Li)
        d = [to_dev(x) for x in (ltf, ltb, lact)]
        capi = int(lact.sum() * rng.choice([0.5, 10.0])) * Mi
        _check_search(B.partition_search_interleaved(*d, Pi, v, Mi, comm, capi, sd, c0, n, all_makespan=True),
                      orc.search_interleaved(ltf, ltb, lact, Pi, v, Mi, comm, capi, sd, c0, c0 + n, nthreads=NCPU),
                      Pi * v - 1)


@pytest.mark.parametrize("seed", range(4))
def test_many_random_sets(orc, seed):
    """pp_sched_many_* on random sets of problems (random shapes, layouts,
    broadcast strides, empty batches, repeated shapes with other strides),
    prepared from an empty plan cache so the batched builder makes every plan
    and table; every output of every problem against the oracle."""
    import torch

    from gpu_helpers import to_dev
    from pipeline_schedule_simulation_gb300 import binding as B
    rng = np.random.default_rng(5000 + seed)
    batches = []
    for _ in range(int(rng.integers(10, 40))):
        policy, P, M, v = _shape(rng)
        n = int(rng.integers(0, 80))
        batches.append(W.random_batch(policy, P, M, v, n, seed=int(rng.integers(1 << 30)), hi=int(rng.choice([5, 60])),
                                      comm_hi=int(rng.integers(0, 5)),
                                      layout="inst_minor" if rng.random() < 0.5 else "inst_major",
                                      pad_to=int(rng.choice([1, 4])), stride_mb_zero=bool(rng.random() < 0.6)))
    batches += [W.random_batch(b.policy, b.P, b.M, b.v, 9, seed=7, hi=9, layout="inst_major") for b in batches[:3]]
    problems = [{"policy": b.policy, "P": b.P, "M": b.M, "v": b.v, "n": b.n, "strides": b.strides,
                 "cost_f": to_dev(b.cost_f), "cost_b": to_dev(b.cost_b), "comm": to_dev(b.comm) if b.n else None,
                 "comm_strides": b.comm_strides} for b in batches]
    B.cache_clear()
    many = B.Many(problems)
    outs = many()
    torch.cuda.synchronize()
    for b, o in zip(batches, outs):
        got = {k: o[k].cpu().numpy() for k in ("makespan", "idle", "bub_num", "bub_den", "peak", "status")}
        ref = run_oracle(orc, b, nthreads=NCPU)
        assert np.array_equal(got["peak"], ref["peak"])
        if b.n:
            assert_same(got, ref)
    many.close()


@pytest.mark.parametrize("seed", range(3))
def test_separate_backward_latency_random(orc, seed):
    """pp_sched_eval_fb (a latency of its own on backward edges) on random
    shapes of every policy, every op time against the oracle."""
    from gpu_helpers import to_dev
    from pipeline_schedule_simulation_gb300 import binding as B
    rng = np.random.default_rng(6000 + seed)
    for _ in range(10):
        policy, P, M, v = _shape(rng)
        n = int(rng.integers(1, 100))
        b = W.random_batch(policy, P, M, v, n, seed=int(rng.integers(1 << 30)), hi=20, comm_hi=5,
                           layout="inst_minor" if rng.random() < 0.5 else "inst_major")
        comm_b = rng.integers(0, 7, b.comm.shape).astype(np.int32)
        out = B.evaluate(b.policy, b.P, b.M, b.v, to_dev(b.cost_f), to_dev(b.cost_b), b.strides, b.n,
                         comm=to_dev(b.comm), comm_strides=b.comm_strides, op_times=True, comm_b=to_dev(comm_b))
        got = {k: t.cpu().numpy() for k, t in out.items()}
        ref = orc.eval_batch(b.policy, b.P, b.M, b.v, b.cost_f, b.cost_b, b.strides, comm=b.comm,
                             comm_strides=b.comm_strides, n=b.n, op_times=True, nthreads=NCPU, comm_b=comm_b)
        assert_same(got, ref, op_times=True)


@pytest.mark.parametrize("seed", range(3))
def test_host_entry_random(orc, seed):
    """pp_sched_eval_host from pinned host buffers on random shapes, batch
    sizes and workspace sizes (from one 32-instance chunk to the whole batch,
    so every chunking and both the one-slot and two-slot paths run); every
    output against the oracle, two calls in a row with the same staging."""
    import torch

    from pipeline_schedule_simulation_gb300 import binding as B
    rng = np.random.default_rng(7000 + seed)
    for _ in range(6):
        policy, P, M, v = _shape(rng)
        n = int(rng.integers(1, 3000))
        lo_ws = int(B.LIB.pp_sched_eval_host_workspace(P, M, v, 32))
        hi_ws = int(B.LIB.pp_sched_eval_host_workspace(P, M, v, n))
        ws = int(rng.choice([lo_ws, (lo_ws + hi_ws) // 2, hi_ws]))
        ws = (ws + 255) // 256 * 256
        staging = {}
        for call in range(2):
            b = W.random_batch(policy, P, M, v, n, seed=int(rng.integers(1 << 30)), hi=30, comm_hi=5)
            hf, hb, hc = (torch.from_numpy(x).pin_memory() for x in (b.cost_f, b.cost_b, b.comm))
            host, _, _ = B.evaluate_host(policy, P, M, v, hf, hb, n, comm=hc, staging=staging, workspace_bytes=ws)
            torch.cuda.synchronize()
            got = {k: t.numpy().copy() for k, t in host.items()}
            assert_same(got, run_oracle(orc, b, nthreads=NCPU))
