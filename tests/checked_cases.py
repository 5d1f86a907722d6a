"""Cases run through the bounds-checked build of the library (imported with
PPSCHED_CHECKED=1 in a process of its own by tests/test_gpu_checked.py):
every evaluator kernel and every search, each compared with the oracle, then
the record of failed checks read.  Prints one JSON line."""
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
import pipeline_schedule_simulation_gb300.workloads as W  # noqa: E402
from gpu_helpers import (assert_same, assert_same_zb, run_gpu, run_gpu_dp, run_gpu_zb, run_oracle,  # noqa: E402
                         run_oracle_dp, run_oracle_zb, to_dev)
from pipeline_schedule_simulation_gb300 import binding as B  # noqa: E402


def main():
    orc = oracle
    n_cases = 0
    # register, split, lane and slot evaluators: GPipe, 1F1B, FIFO, interleaved,
    # both layouts, costs per microbatch and shared by all microbatches,
    # batches that fill whole warps and ragged ones
    for policy, P, M, v in ((W.ONEF1B, 8, 16, 1), (W.GPIPE, 4, 8, 1), (W.GPIPE_FIFO, 3, 7, 1),
                            (W.ONEF1B, 16, 20, 1), (W.INTERLEAVED, 4, 8, 2), (W.INTERLEAVED, 8, 16, 4),
                            (W.INTERLEAVED, 3, 9, 3)):
        for layout in ("inst_minor", "inst_major"):
            for n, mbz in ((77, False), (161, True), (1024, False)):
                b = W.random_batch(policy, P, M, v, n, seed=n + P + M, hi=12, comm_hi=5, layout=layout,
                                   stride_mb_zero=mbz)
                assert_same(run_gpu(b, op_times=True), run_oracle(orc, b, op_times=True), op_times=True)
                n_cases += 1
    # a backward latency of its own (the lane evaluator for every policy)
    for policy, P, M, v in ((W.ONEF1B, 8, 16, 1), (W.INTERLEAVED, 4, 8, 2)):
        b = W.random_batch(policy, P, M, v, 130, seed=4 + P, hi=12, comm_hi=6, pad_to=4)
        cb = np.random.default_rng(P).integers(0, 9, size=b.comm.shape).astype(np.int32)
        out = B.evaluate(policy, P, M, v, to_dev(b.cost_f), to_dev(b.cost_b), b.strides, b.n, comm=to_dev(b.comm),
                         comm_strides=b.comm_strides, op_times=True, comm_b=to_dev(cb))
        torch.cuda.synchronize()
        g = {k: t.cpu().numpy() for k, t in out.items()}
        r = orc.eval_batch(policy, P, M, v, b.cost_f, b.cost_b, b.strides, comm=b.comm,
                           comm_strides=b.comm_strides, n=b.n, op_times=True, nthreads=8, comm_b=cb)
        assert_same(g, r, op_times=True)
        n_cases += 1
    # many problems in fused launches (costs shared by all microbatches)
    probs, refs = [], []
    for policy, P, M, v in ((W.ONEF1B, 4, 8, 1), (W.INTERLEAVED, 4, 8, 2), (W.GPIPE, 3, 5, 1)):
        b = W.random_batch(policy, P, M, v, 40, seed=P + M, hi=12, comm_hi=3, stride_mb_zero=True)
        probs.append(dict(policy=policy, P=P, M=M, v=v, cost_f=to_dev(b.cost_f), cost_b=to_dev(b.cost_b),
                          strides=b.strides, n=b.n, comm=to_dev(b.comm), comm_strides=b.comm_strides))
        refs.append(run_oracle(orc, b))
    many = B.Many(probs)
    outs = many()
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert_same({k: t.cpu().numpy() for k, t in o.items()}, r)
        n_cases += 1
    many.close()
    # Zero Bubble and DualPipe
    for policy in (W.ZB1P, W.ZB2P):
        b = W.random_zb(policy, 8, 12, 90, seed=policy, hi=12, w_hi=9, comm_hi=5)
        assert_same_zb(run_gpu_zb(b, op_times=True), run_oracle_zb(orc, b, op_times=True), op_times=True)
        n_cases += 1
    b = W.random_batch(W.ONEF1B, 8, 12, 1, 90, seed=9, lo=1, hi=12, comm_hi=5)
    assert_same_zb(run_gpu_dp(b, 5, op_times=True), run_oracle_dp(orc, b, 5, op_times=True), op_times=True)
    n_cases += 1
    # the three searches on a small model, every candidate's makespan
    rng = np.random.default_rng(11)
    L, P, M = 24, 4, 8
    ltf = rng.integers(1, 20, L).astype(np.int32)
    ltb = rng.integers(1, 40, L).astype(np.int32)
    lact = rng.integers(1, 4, L).astype(np.int64)
    cap = int(3 * lact.sum())
    dev = [to_dev(x) for x in (ltf, ltb, lact)]
    g = B.partition_search(*dev, P, M, 1, cap, 77, 0, 500, all_makespan=True)
    r = orc.search(ltf, ltb, lact, P, M, 1, cap, 77, 0, 500, nthreads=8)
    assert np.array_equal(g["all_makespan"].cpu().numpy(), r["all_makespan"])
    total = int(orc.binom(L - 1, P - 1))
    g = B.partition_search_ranks(*dev, P, M, 1, cap, 0, total, all_makespan=True)
    r = orc.search_ranks(ltf, ltb, lact, P, M, 1, cap, 0, total, nthreads=8)
    assert np.array_equal(g["all_makespan"].cpu().numpy(), r["all_makespan"])
    g = B.partition_search_interleaved(*dev, P, 2, M, 1, cap, 78, 0, 300, all_makespan=True)
    r = orc.search_interleaved(ltf, ltb, lact, P, 2, M, 1, cap, 78, 0, 300, nthreads=8)
    assert np.array_equal(g["all_makespan"].cpu().numpy(), r["all_makespan"])
    n_cases += 3
    torch.cuda.synchronize()
    checked, word = B.debug_checks()
    print(json.dumps({"lib": os.path.basename(B.build_lib.LIB_CHECKED), "checked": checked, "failure": word,
                      "cases": n_cases}))


if __name__ == "__main__":
    main()
