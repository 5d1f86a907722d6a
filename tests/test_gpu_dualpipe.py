"""GPU DualPipe evaluator (pp_sched_eval_dualpipe) against the oracle's
DualPipe simulation: every output bit-exact, including every op's start and
end and the per-instance peak of held activations."""
import os

import numpy as np
import pytest
import torch

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import assert_same_zb, run_gpu, run_gpu_dp, run_oracle_dp, to_dev

pytestmark = pytest.mark.gpu

NCPU = os.cpu_count() or 8

SHAPES = [(1, 1, 1), (1, 5, 2), (2, 4, 2), (2, 7, 0), (2, 7, 7), (3, 6, 3), (4, 8, 4), (4, 9, 6), (5, 13, 6),
          (8, 16, 8), (8, 64, 32), (8, 20, 3), (12, 30, 15), (16, 40, 20), (16, 9, 4), (7, 3, 1)]


@pytest.mark.parametrize("P,M,m_a", SHAPES)
@pytest.mark.parametrize("layout", ["inst_minor", "inst_major"])
@pytest.mark.parametrize("cap1", [None, 0, 5])
def test_random_batches_every_op(orc, monkeypatch, P, M, m_a, layout, cap1):
    """Every op time against the oracle, with the kernel's first phase as
    configured (None), skipped (0: every instance on the common-tick phase)
    and cut short (5 steps: instances handed over part-way)."""
    if cap1 is not None:
        monkeypatch.setenv("PPSCHED_DP_PHASE1_STEPS", str(cap1))
    for n in (37, 133):
        b = W.random_batch(W.ONEF1B, P, M, 1, n, seed=P * 100 + M + n, lo=1, hi=9, comm_hi=4, layout=layout)
        g = run_gpu_dp(b, m_a, op_times=True)
        r = run_oracle_dp(orc, b, m_a, op_times=True, nthreads=NCPU)
        assert_same_zb(g, r, op_times=True)
        assert (g["status"] == 0).all()


@pytest.mark.parametrize("layout", ["inst_minor", "inst_major"])
def test_costs_shared_by_microbatches(orc, layout):
    """Costs per (block) only, broadcast over microbatches (stride 0)."""
    for P, M, m_a in ((4, 12, 6), (8, 17, 9), (16, 9, 0)):
        b = W.random_batch(W.ONEF1B, P, M, 1, 101, seed=P + M, lo=1, hi=9, layout=layout, stride_mb_zero=True)
        assert b.strides[2] == 0
        g = run_gpu_dp(b, m_a, op_times=True)
        r = run_oracle_dp(orc, b, m_a, op_times=True, nthreads=NCPU)
        assert_same_zb(g, r, op_times=True)


def test_one_route_is_the_1f1b_evaluator(orc):
    """All microbatches on route A is 1F1B: the same makespans, idle ticks and
    bubble pairs as pp_sched_eval's 1F1B kernel."""
    b = W.hetero_1f1b(n=4096, seed=9)
    g = run_gpu_dp(b, b.M)
    h = run_gpu(b)
    for k in ("makespan", "idle", "bub_num", "bub_den", "status"):
        assert np.array_equal(g[k], h[k]), k


def test_statuses(orc):
    P, M, n = 4, 6, 40
    b = W.random_batch(W.ONEF1B, P, M, 1, n, seed=5, lo=1, hi=9, layout="inst_major")
    cf = b.cost_f.reshape(n, P, M)
    cb = b.cost_b.reshape(n, P, M)
    cm = b.comm.reshape(n, P - 1)
    cf[3, 2, 5] = -1
    cm[4, 0] = -3
    cb[7, 1, 1] = 0
    cf[9, 0, 0] = 2**31 - 9
    cb[10, 3, 5] = 2**30
    cf[10, 3, 5] = 2**30
    g = run_gpu_dp(b, 3)
    r = run_oracle_dp(orc, b, 3)
    assert g["status"][3] == 1 and g["status"][4] == 1
    assert g["status"][7] == 3 and g["status"][9] == 2 and g["status"][10] == 2
    assert_same_zb(g, r)


@pytest.mark.parametrize("cap1", [None, 0, 40])
def test_hetero_full_batch(orc, monkeypatch, cap1):
    """65,536 heterogeneous instances (P=8, M=64, 32 microbatches per route):
    every instance against the oracle, and the page's peak of at most p+1;
    with the first phase as configured, skipped, and cut short."""
    if cap1 is not None:
        monkeypatch.setenv("PPSCHED_DP_PHASE1_STEPS", str(cap1))
    b = W.hetero_dualpipe()
    m_a = b.meta["m_a"]
    g = run_gpu_dp(b, m_a)
    assert (g["status"] == 0).all()
    r = run_oracle_dp(orc, b, m_a, nthreads=NCPU)
    assert_same_zb(g, r)
    assert (g["peak"] <= b.P + 1).all()


def test_argument_errors():
    from pipeline_schedule_simulation_gb300 import binding as B
    x = torch.ones(64, dtype=torch.int32, device="cuda")
    with pytest.raises(B.PPSchedError):
        B.evaluate_dualpipe(17, 4, 2, x, x, (4, 2, 1), 2)
    with pytest.raises(B.PPSchedError):
        B.evaluate_dualpipe(4, 4, 5, x, x, (4, 2, 1), 2)
    out = B.evaluate_dualpipe(2, 2, 1, x, x, (4, 2, 1), 0)
    assert out["makespan"].numel() == 0
