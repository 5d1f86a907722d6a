"""GPU Zero Bubble evaluator (pp_sched_eval_zb) against the oracle's ZB
simulator: every output bit-exact, including per-op times and the per-instance
peak of held microbatches."""
import os

import numpy as np
import pytest
import torch

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import assert_same_zb, run_gpu_zb, run_oracle_zb, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (1, 5), (2, 2), (2, 7), (3, 3), (3, 10), (4, 8), (5, 4), (6, 13), (8, 8), (8, 21),
          (12, 6), (16, 16), (16, 40)]


@pytest.mark.parametrize("policy", [W.ZB1P, W.ZB2P])
@pytest.mark.parametrize("P,M", SHAPES)
@pytest.mark.parametrize("layout", ["inst_minor", "inst_major"])
def test_random_batches(orc, policy, P, M, layout):
    # several warps and a ragged last warp; W often free (0) to exercise
    # repeated decisions at one tick
    for n, seed, w_hi in ((37, 1, 9), (70, 2, 2)):
        batch = W.random_zb(policy, P, M, n, seed=seed + 10 * P + M, hi=12, w_hi=w_hi, comm_hi=5, layout=layout)
        g = run_gpu_zb(batch, op_times=True)
        r = run_oracle_zb(orc, batch, op_times=True)
        assert (r["status"] == 0).all()
        assert_same_zb(g, r, op_times=True)


@pytest.mark.parametrize("policy", [W.ZB1P, W.ZB2P])
def test_w_heavy_and_w_free(orc, policy):
    """W much longer than F and B (the budget binds), and W of zero cost."""
    for seed, (wlo, whi) in ((3, (20, 60)), (4, (0, 0))):
        batch = W.random_zb(policy, 6, 24, 50, seed=seed, lo=1, hi=6, w_lo=wlo, w_hi=whi, comm_hi=3)
        g = run_gpu_zb(batch, op_times=True)
        r = run_oracle_zb(orc, batch, op_times=True)
        assert_same_zb(g, r, op_times=True)
        L = 6 if policy == W.ZB1P else 12
        assert (g["peak"] <= L).all()


def test_zb1p_without_w_equals_1f1b_evaluator(B):
    """With W free, ZB1P's makespan equals the 1F1B evaluator's (a different
    kernel) on the same F and B costs."""
    batch = W.random_zb(W.ZB1P, 8, 16, 300, seed=5, lo=1, hi=30, w_lo=0, w_hi=0, comm_hi=4)
    g = run_gpu_zb(batch)
    out = B.evaluate(W.ONEF1B, 8, 16, 1, to_dev(batch.cost_f), to_dev(batch.cost_b), batch.strides, batch.n,
                     comm=to_dev(batch.comm), comm_strides=batch.comm_strides)
    torch.cuda.synchronize()
    assert np.array_equal(g["makespan"], out["makespan"].cpu().numpy())


@pytest.fixture(scope="module")
def B():
    from pipeline_schedule_simulation_gb300 import binding
    return binding


def test_statuses(orc, B):
    P, M, n = 4, 6, 40
    batch = W.random_zb(W.ZB1P, P, M, n, seed=9, layout="inst_major")
    cf = batch.cost_f.reshape(n, P, M)
    cb = batch.cost_b.reshape(n, P, M)
    cw = batch.cost_w.reshape(n, P, M)
    cf[1, 2, 3] = -2          # negative F
    cw[2, 0, 0] = -1          # negative W
    cb[3, 1, 1] = 0           # zero B
    cf[4, 3, 5] = 0           # zero F
    batch.comm.reshape(n, P - 1)[5, 2] = -3      # negative comm
    cb[6, 0, 5] = 2**31 - 10  # overflow
    cf[7, 0, 0] = 0
    cw[7, 1, 1] = -5          # negative beats zero
    g = run_gpu_zb(batch)
    r = run_oracle_zb(orc, batch)
    want = {1: B.ST_NEG_COST, 2: B.ST_NEG_COST, 3: B.ST_ZERO_COST, 4: B.ST_ZERO_COST, 5: B.ST_NEG_COST,
            6: B.ST_OVERFLOW, 7: B.ST_NEG_COST}
    for x, st in want.items():
        assert g["status"][x] == st, x
    assert_same_zb(g, r)


def test_broadcast_strides(orc):
    """Costs shared by every instance and microbatch (strides 0)."""
    P, M, n = 5, 9, 33
    rng = np.random.default_rng(2)
    cf = rng.integers(1, 9, P).astype(np.int32)
    cb = rng.integers(1, 9, P).astype(np.int32)
    cw = rng.integers(0, 9, P).astype(np.int32)
    cm = rng.integers(0, 4, (n, P - 1)).astype(np.int32)
    for policy in (W.ZB1P, W.ZB2P):
        batch = W.Batch(policy, P, M, 1, n, cf, cb, (0, 1, 0), cm.reshape(-1), (P - 1, 1), cost_w=cw)
        g = run_gpu_zb(batch, op_times=True)
        r = run_oracle_zb(orc, batch, op_times=True)
        assert_same_zb(g, r, op_times=True)


@pytest.mark.parametrize("policy", [W.ZB1P, W.ZB2P])
def test_hetero_full_batch(orc, policy):
    """65,536 heterogeneous instances (P=8, M=64): every instance against the
    oracle, plus invariants."""
    batch = W.hetero_zb(policy)
    g = run_gpu_zb(batch)
    assert (g["status"] == 0).all()
    r = run_oracle_zb(orc, batch, nthreads=os.cpu_count() or 8)
    assert_same_zb(g, r)
    busy = np.zeros((batch.n, 8), np.int64)
    for c in (batch.cost_f, batch.cost_b, batch.cost_w):
        busy += c.reshape(8, 64, batch.n).sum(axis=1).T
    assert np.array_equal(g["idle"].astype(np.int64), g["makespan"][:, None].astype(np.int64) - busy)
    assert np.array_equal(g["bub_den"], 8 * g["makespan"].astype(np.int64))
    assert (g["peak"] <= (8 if policy == W.ZB1P else 16)).all()


def test_argument_errors(B):
    x = torch.ones(64, dtype=torch.int32, device="cuda")
    with pytest.raises(B.PPSchedError):
        B.evaluate_zb(W.ONEF1B, 2, 2, x, x, x, (4, 2, 1), 2)
    with pytest.raises(B.PPSchedError):
        B.evaluate_zb(W.ZB1P, 17, 2, x, x, x, (4, 2, 1), 2)
    out = B.evaluate_zb(W.ZB1P, 2, 2, x, x, x, (4, 2, 1), 0)
    assert out["makespan"].numel() == 0
