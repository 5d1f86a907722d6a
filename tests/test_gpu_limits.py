"""Every GPU entry point at the library's declared limits, against the oracle.

The limits (ppsched.h): P <= PP_MAX_P = 16 devices, P*v <= PP_MAX_S = 64
virtual stages, M*v <= PP_MAX_MV = 32,768 (65,536 ops per device), and in the
searches L <= 256 layers with C(L-1, S-1) below 2^64.  Each case sits on one or
more of them at once, with a ragged batch where the kernel works in warps of
instances, and compares every output (per-op times included) bit for bit.
The refusals one step past each limit are host-side and tested without a GPU
(test_abi.py).  Zero Bubble and DualPipe sit at P = 16 and M = 32,768.
"""
import numpy as np
import pytest
import torch

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import (assert_same, assert_same_zb, run_gpu, run_gpu_dp, run_gpu_zb, run_oracle, run_oracle_dp,
                         run_oracle_zb, to_dev)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("policy,P,M,v,n,layout", [
    (W.ONEF1B, 16, 32768, 1, 37, "inst_minor"),       # P and M*v at the limit, 65,536 ops per device
    (W.GPIPE, 16, 32768, 1, 5, "inst_major"),         # peak = M = 32,768
    (W.GPIPE_FIFO, 16, 32768, 1, 3, "inst_minor"),
    (W.INTERLEAVED, 16, 8192, 4, 9, "inst_minor"),    # P, P*v = 64 and M*v at the limit
    (W.INTERLEAVED, 8, 4096, 8, 5, "inst_major"),     # v = 8: 64 virtual stages on 8 devices
])
def test_eval_at_limits(orc, policy, P, M, v, n, layout):
    batch = W.random_batch(policy, P, M, v, n, seed=P + M + v, hi=30, comm_hi=6, layout=layout)
    g = run_gpu(batch, op_times=True)
    r = run_oracle(orc, batch, op_times=True)
    assert (r["status"] == 0).all()
    assert_same(g, r, op_times=True)


@pytest.mark.parametrize("policy", [W.ZB1P, W.ZB2P])
def test_zero_bubble_at_limits(orc, policy):
    """P = 16 and M = 32,768 (98,304 F, B and W ops per device)."""
    batch = W.random_zb(policy, 16, 32768, 2, seed=3 + policy, hi=30, w_hi=30, comm_hi=6)
    g = run_gpu_zb(batch, op_times=True)
    r = run_oracle_zb(orc, batch, op_times=True, nthreads=2)
    assert (r["status"] == 0).all()
    assert_same_zb(g, r, op_times=True)


@pytest.mark.parametrize("m_a", [16384, 32768, 0, 1])
def test_dualpipe_at_limits(orc, m_a):
    """P = 16 and M = 32,768 (65,536 F and B ops per device): both routes
    half full, every microbatch on route A, every one on route B, and a
    single one on route A."""
    batch = W.random_batch(W.ONEF1B, 16, 32768, 1, 2, seed=71 + m_a % 7, lo=1, hi=30, comm_hi=6)
    g = run_gpu_dp(batch, m_a, op_times=True)
    r = run_oracle_dp(orc, batch, m_a, op_times=True, nthreads=2)
    assert (r["status"] == 0).all()
    assert_same_zb(g, r, op_times=True)


def _layers(L, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(1, 20, L).astype(np.int32), rng.integers(1, 40, L).astype(np.int32),
            rng.integers(1, 4, L).astype(np.int64))


def test_searches_at_limits(orc):
    """The searches at their largest shapes: P = 16 stages at M = 32,768 with
    L = 131 layers, the most whose C(130, 15) = 1.69e19 splits fit 64 bits (so
    SplitMix64's output is reduced modulo a number near 2^64 and the unranking
    walks binomials near 2^64); exhaustive ranks just below 2^63, the largest an
    int64 rank can name; L = 256 layers into 4 stages; and 64 interleaved
    ranges (P = 16, v = 4, M*v = 32,768) of L = 84 layers, the most for S = 64."""
    from pipeline_schedule_simulation_gb300 import binding as B
    seed, cap = 987654321, 10**12
    cases = []
    ltf, ltb, lact = _layers(131, 41)
    d = [to_dev(x) for x in (ltf, ltb, lact)]
    cases.append((B.partition_search(*d, 16, 32768, 1, cap, seed, 5, 24, all_makespan=True),
                  orc.search(ltf, ltb, lact, 16, 32768, 1, cap, seed, 5, 29, nthreads=8), 15))
    r0 = (1 << 63) - 30
    cases.append((B.partition_search_ranks(*d, 16, 32768, 1, cap, r0, 24, all_makespan=True),
                  orc.search_ranks(ltf, ltb, lact, 16, 32768, 1, cap, r0, r0 + 24, nthreads=8), 15))
    ltf, ltb, lact = _layers(256, 42)
    d = [to_dev(x) for x in (ltf, ltb, lact)]
    cases.append((B.partition_search(*d, 4, 32768, 2, cap, seed, 0, 24, all_makespan=True),
                  orc.search(ltf, ltb, lact, 4, 32768, 2, cap, seed, 0, 24, nthreads=8), 3))
    ltf, ltb, lact = _layers(84, 43)
    d = [to_dev(x) for x in (ltf, ltb, lact)]
    cases.append((B.partition_search_interleaved(*d, 16, 4, 8192, 1, cap, seed, 3, 8, all_makespan=True),
                  orc.search_interleaved(ltf, ltb, lact, 16, 4, 8192, 1, cap, seed, 3, 11, nthreads=8), 63))
    torch.cuda.synchronize()
    for got, ref, k in cases:
        assert (ref["all_makespan"] > 0).all()
        assert np.array_equal(got["all_makespan"].cpu().numpy(), ref["all_makespan"])
        assert int(got["best_idx"].item()) == ref["best_idx"]
        assert int(got["best_makespan"].item()) == ref["best_makespan"]
        assert list(got["best_cuts"].cpu().numpy()) == list(ref["first"][1:k + 1])
