"""Host threads calling the library at once, each on its own stream: new
shapes (plans built concurrently), new stride pairs (kernel tables built
concurrently), several evaluator kernels and the many-problem path; every
result against the oracle.  ctypes releases the interpreter lock during a
library call, so the calls really overlap."""
import threading

import numpy as np
import pytest
import torch

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import assert_same, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def test_threads_share_the_plan_cache(orc):
    from pipeline_schedule_simulation_gb300 import binding as B
    # shapes the other tests do not use, so the threads build their plans
    shapes = [(W.ONEF1B, 7, 53, 1), (W.GPIPE, 11, 47, 1), (W.INTERLEAVED, 5, 35, 3), (W.ONEF1B, 13, 61, 1),
              (W.GPIPE_FIFO, 9, 59, 1), (W.INTERLEAVED, 6, 42, 2), (W.ONEF1B, 2, 97, 1), (W.GPIPE, 15, 43, 1)]
    jobs = []
    for t in range(4):
        for i, (policy, P, M, v) in enumerate(shapes):
            # every thread evaluates every shape, in its own order, in both
            # layouts and with costs per microbatch or shared
            layout = "inst_minor" if (t + i) % 2 == 0 else "inst_major"
            b = W.random_batch(policy, P, M, v, 97 + 13 * t, seed=100 * t + i, hi=15, comm_hi=4, layout=layout,
                               stride_mb_zero=(t + i) % 3 == 0, pad_to=1 + 3 * ((t + i) % 2))
            jobs.append((t, b))
    errors, results = [], {}
    barrier = threading.Barrier(4)

    def worker(t):
        try:
            s = torch.cuda.Stream()
            mine = [(k, b) for k, (tt, b) in enumerate(jobs) if tt == t]
            if t % 2:
                mine.reverse()
            dev = {k: (to_dev(b.cost_f), to_dev(b.cost_b), to_dev(b.comm)) for k, b in mine}
            torch.cuda.synchronize()
            barrier.wait()
            with torch.cuda.stream(s):
                for k, b in mine:
                    f, g, c = dev[k]
                    results[k] = B.evaluate(b.policy, b.P, b.M, b.v, f, g, b.strides, b.n, comm=c,
                                            comm_strides=b.comm_strides, op_times=True, stream=s)
            s.synchronize()
        except Exception as e:  # reported below, with the thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for k, (t, b) in enumerate(jobs):
        g = {key: v.cpu().numpy() for key, v in results[k].items()}
        assert_same(g, run_oracle(orc, b, op_times=True), op_times=True)
