"""pp_sched_many_*: many problems with their own shapes in a few launches.

Every output of every problem must equal pp_sched_eval's on the same inputs
and the oracle's: over the whole closed-form sweep (4,139 shapes, all taken by
the fused kernels), over a mixed set where some problems are fused and the
rest go through pp_sched_eval, after the cost tables are rewritten in place,
for the per-instance statuses, and when the fused launches are replayed from
a CUDA graph.
"""
import os

import numpy as np
import pytest
import torch

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import assert_same, run_oracle, to_dev

pytestmark = pytest.mark.gpu

KEYS = ("makespan", "idle", "bub_num", "bub_den", "peak", "status")


def _problem(b):
    return {"policy": b.policy, "P": b.P, "M": b.M, "v": b.v, "n": b.n, "strides": b.strides,
            "cost_f": to_dev(b.cost_f), "cost_b": to_dev(b.cost_b),
            "comm": to_dev(b.comm) if b.n else None, "comm_strides": b.comm_strides}


def _fill(out, value):
    for t in out.values():
        t.fill_(value)


def _single(B, q):
    """pp_sched_eval on one problem's device tensors."""
    o = B.evaluate(q["policy"], q["P"], q["M"], q["v"], q["cost_f"], q["cost_b"], q["strides"], q["n"],
                   comm=q["comm"], comm_strides=q["comm_strides"])
    return {k: o[k].cpu().numpy() for k in KEYS}


def _host(out):
    return {k: out[k].cpu().numpy() for k in KEYS}


def test_closed_form_sweep_fused(orc):
    """The whole sweep in one prepared set, its plans and tables built from an
    empty cache in one batch: every problem fused, a handful of launches,
    every output of every problem equal to pp_sched_eval's and to the
    oracle's."""
    from pipeline_schedule_simulation_gb300 import binding as B
    shapes = W.sweep_shapes()
    batches = [W.sweep_batch(*s) for s in shapes]
    problems = [_problem(b) for b in batches]
    B.cache_clear()  # every plan and table is built by the preparation's batched build
    many = B.Many(problems)
    info = many.info()
    assert info == {"fused_problems": len(shapes), "launches": info["launches"], "other_problems": 0}
    assert 1 <= info["launches"] <= 6
    for q in many.problems:
        _fill(q["out"], -3)
    outs = many()
    torch.cuda.synchronize()
    for i, (b, q, o) in enumerate(zip(batches, problems, outs)):
        got = _host(o)
        want = _single(B, q)
        for k in KEYS:
            assert np.array_equal(got[k], want[k]), (shapes[i], k)
        assert_same(got, run_oracle(orc, b, nthreads=os.cpu_count() or 8))
    many.close()


MIXED = [  # (policy, P, M, v, n, layout, stride_mb_zero)
    (W.ONEF1B, 8, 64, 1, 161, "inst_minor", True), (W.ONEF1B, 8, 64, 1, 77, "inst_minor", False),
    (W.GPIPE, 4, 12, 1, 33, "inst_major", True), (W.GPIPE_FIFO, 16, 9, 1, 70, "inst_minor", True),
    (W.ONEF1B, 1, 7, 1, 5, "inst_minor", True), (W.GPIPE, 3, 1, 1, 1, "inst_major", True),
    (W.ONEF1B, 12, 20, 1, 0, "inst_minor", True), (W.ONEF1B, 16, 40, 1, 129, "inst_major", True),
    (W.INTERLEAVED, 4, 8, 2, 161, "inst_minor", True), (W.INTERLEAVED, 8, 16, 4, 70, "inst_major", True),
    (W.INTERLEAVED, 16, 32, 2, 31, "inst_minor", True), (W.INTERLEAVED, 3, 9, 3, 77, "inst_minor", False),
    (W.INTERLEAVED, 1, 3, 5, 9, "inst_minor", True), (W.GPIPE, 5, 13, 1, 200, "inst_minor", False),
]


def test_mixed_problems_and_rewrites(orc):
    """Fused and unfused problems in one set (costs per microbatch, an empty
    batch), against the oracle; then the cost tables are rewritten in place and
    the same handle evaluates the new values."""
    from pipeline_schedule_simulation_gb300 import binding as B
    batches = [W.random_batch(p, P, M, v, n, seed=7 * P + M + n, hi=15, comm_hi=4, layout=lay, stride_mb_zero=z)
               for p, P, M, v, n, lay, z in MIXED]
    problems = [_problem(b) for b in batches]
    many = B.Many(problems)
    info = many.info()
    assert info["fused_problems"] == sum(1 for m in MIXED if m[6] and m[4] > 0)
    assert info["other_problems"] == len(MIXED) - info["fused_problems"]
    for round_ in range(2):
        for q in many.problems:
            _fill(q["out"], -3)
        outs = many()
        torch.cuda.synchronize()
        for b, o in zip(batches, outs):
            got = _host(o)
            ref = run_oracle(orc, b)
            assert np.array_equal(got["peak"], ref["peak"])
            if b.n:
                assert_same(got, ref)
        # new costs, same buffers
        rng = np.random.default_rng(100 + round_)
        for b, q in zip(batches, many.problems):
            if not b.n:
                continue
            b.cost_f[...] = rng.integers(0, 15, b.cost_f.shape, dtype=np.int32)
            b.cost_b[...] = rng.integers(0, 15, b.cost_b.shape, dtype=np.int32)
            q["cost_f"].copy_(torch.from_numpy(b.cost_f))
            q["cost_b"].copy_(torch.from_numpy(b.cost_b))
    many.close()


def test_statuses_through_the_fused_kernels(orc):
    """A negative cost, a negative comm and an int32 overflow in fused
    problems are flagged per instance as pp_sched_eval and the oracle flag
    them; the other instances are exact."""
    from pipeline_schedule_simulation_gb300 import binding as B
    batches = []
    for p, P, M, v in ((W.ONEF1B, 8, 16, 1), (W.GPIPE, 4, 8, 1), (W.INTERLEAVED, 4, 8, 2)):
        b = W.random_batch(p, P, M, v, 40, seed=P + M, hi=12, comm_hi=3, stride_mb_zero=True)
        cf = b.cost_f.reshape(P * v, 1, 40)
        cf[1, 0, 3] = -1                        # instance 3: negative cost
        b.comm.reshape(-1, 40)[0, 7] = -2       # instance 7: negative comm
        cf[:, 0, 11] = 2**30                    # instance 11: ticks beyond int32
        batches.append(b)
    problems = [_problem(b) for b in batches]
    many = B.Many(problems)
    assert many.info()["fused_problems"] == 3
    outs = many()
    torch.cuda.synchronize()
    for b, q, o in zip(batches, problems, outs):
        got, ref = _host(o), run_oracle(orc, b)
        assert set(np.nonzero(ref["status"])[0]) == {3, 7, 11}
        assert_same(got, ref)
        want = _single(B, q)
        assert np.array_equal(got["status"], want["status"])
    many.close()


def test_fused_launches_in_a_cuda_graph():
    """A set that is fused entirely only launches kernels: captured once in a
    CUDA graph, each replay rewrites the outputs with the same values."""
    from pipeline_schedule_simulation_gb300 import binding as B
    shapes = [s for s in W.sweep_shapes() if s[1] in (2, 7, 16) and s[2] % 9 == 0]
    problems = [_problem(W.sweep_batch(*s)) for s in shapes]
    many = B.Many(problems)
    assert many.info()["other_problems"] == 0
    ref = [_host(o) for o in many()]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        many(stream=side)
    for _ in range(2):
        for q in many.problems:
            _fill(q["out"], -9)
        graph.replay()
        torch.cuda.synchronize()
        for q, r in zip(many.problems, ref):
            got = _host(q["out"])
            for k in KEYS:
                assert np.array_equal(got[k], r[k])
    many.close()
