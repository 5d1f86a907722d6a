"""pp_sched_eval_noalloc — the evaluation entry point that allocates nothing.

It serves callers that cannot let a library call cudaMalloc (their device
memory belongs to another allocator, or must not grow while they run).  These
tests call it through the C ABI and check every output against pp_sched_eval,
bit for bit, and against the CPU oracle, instance by instance, on a sequence
of calls that walks every state of the library's fixed table array:

  1. a new shape: the tables are built in the array;
  2. the same shape and strides with new costs: the tables are reused as they
     are (nothing rebuilt, one launch);
  3. the same shape with another stride pair (rows padded to a multiple of 8
     instances): only the stride-dependent kernel tables are rebuilt;
  4. another shape and layout: everything is rebuilt;
  5. the first shape again: rebuilt once more, then reused by a sixth call.

The file is collected last on purpose and depends on no other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import assert_same, run_oracle

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _outs(n, P):
    return {"makespan": torch.full((n,), -7, dtype=torch.int32, device="cuda"),
            "idle": torch.full((n, P), -7, dtype=torch.int32, device="cuda"),
            "bub_num": torch.full((n,), -7, dtype=torch.int64, device="cuda"),
            "bub_den": torch.full((n,), -7, dtype=torch.int64, device="cuda"),
            "peak": torch.full((P,), -7, dtype=torch.int32, device="cuda"),
            "status": torch.full((n,), -7, dtype=torch.int8, device="cuda")}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(B, b, cf, cb, cm):
    o = _outs(b.n, b.P)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = B.LIB.pp_sched_eval_noalloc(b.policy, b.P, b.M, _p(cf), _p(cb), *b.strides, _p(cm), *b.comm_strides,
                                     b.n, _p(o["makespan"]), _p(o["idle"]), _p(o["bub_num"]),
                                     _p(o["bub_den"]), _p(o["peak"]), _p(o["status"]), stream)
    assert rc == B.PP_OK, B.status_str(rc)
    return o


def _reference(B, b, cf, cb, cm):
    o = _outs(b.n, b.P)
    B.evaluate(b.policy, b.P, b.M, 1, cf, cb, b.strides, b.n, comm=cm, comm_strides=b.comm_strides, out=o)
    return o


def _same(x, y):
    torch.cuda.synchronize()
    for k in x:
        assert torch.equal(x[k].cpu(), y[k].cpu()), k


def test_noalloc_matches_eval_and_oracle_on_consecutive_calls(orc):
    from pipeline_schedule_simulation_gb300 import binding as B
    P, M = 8, 64
    calls = [
        ("new shape", W.hetero_1f1b(n=5004, seed=21)),
        ("same shape and strides, new costs", W.hetero_1f1b(n=5004, seed=22)),
        ("same shape, rows padded to 8", W.random_batch(W.ONEF1B, P, M, 1, 5001, seed=23, lo=1, hi=200,
                                                        pad_to=8)),
        ("another shape and layout", W.random_batch(W.GPIPE, 4, 16, 1, 777, seed=24, hi=30,
                                                    layout="inst_major")),
        ("first shape again", W.hetero_1f1b(n=5004, seed=25)),
        ("first shape, reused", W.hetero_1f1b(n=5004, seed=26)),
    ]
    assert calls[0][1].strides != calls[2][1].strides      # a different stride pair at the same shape
    for what, b in calls:
        cf, cb, cm = _dev(b.cost_f), _dev(b.cost_b), _dev(b.comm)
        got = _noalloc(B, b, cf, cb, cm)
        want = _reference(B, b, cf, cb, cm)
        _same(got, want)
        g = {k: v.cpu().numpy() for k, v in got.items()}
        assert (g["status"] == 0).all(), what
        assert_same(g, run_oracle(orc, b, nthreads=8))


def test_noalloc_rejects_what_it_does_not_cover():
    from pipeline_schedule_simulation_gb300 import binding as B
    L = B.LIB
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    x = torch.zeros(64, dtype=torch.int32, device="cuda")
    # interleaved 1F1B is not served by this entry point
    assert L.pp_sched_eval_noalloc(B.INTERLEAVED, 4, 8, _p(x), _p(x), 1, 0, 0, None, 0, 0, 4,
                                   None, None, None, None, None, None, s) == B.PP_ERR_ARG
    # a shape whose tables exceed the fixed array: P=16, M=32768 needs 1M ops
    assert L.pp_sched_eval_noalloc(B.ONEF1B, 16, 32768, _p(x), _p(x), 1, 0, 0, None, 0, 0, 4,
                                   None, None, None, None, None, None, s) == B.PP_ERR_SIZE
