"""The C-ABI library loads without a GPU and exports every declared entry
point; host-side argument checks answer before any CUDA call."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(pp_sched_\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from pipeline_schedule_simulation_gb300 import build_lib
    build_lib.build()
    return ctypes.CDLL(build_lib.LIB)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "pp_sched_eval" in names and "pp_sched_plan" in names
    for name in names:
        assert hasattr(lib, name), name


def test_binding_exports_match_header():
    from pipeline_schedule_simulation_gb300 import binding
    assert sorted(binding.EXPORTS) == _declared()


def test_host_argument_errors_without_gpu():
    from pipeline_schedule_simulation_gb300 import binding as B
    L = B.LIB
    nul = None
    def ev(pol, P, M, v, n=4, f=1, b=1, si=1):
        return L.pp_sched_eval(pol, P, M, v, f, b, si, 0, 0, nul, 0, 0, n, nul, nul, nul, nul,
                               nul, nul, nul, 0, 0, nul, nul)
    assert ev(9, 4, 8, 1) == B.PP_ERR_ARG           # unknown policy
    assert ev(B.ZB1P, 4, 8, 1) == B.PP_ERR_ARG      # Zero Bubble needs pp_sched_eval_zb
    assert ev(B.ZB2P, 4, 8, 1) == B.PP_ERR_ARG
    assert ev(B.GPIPE_FIFO, 4, 8, 2) == B.PP_ERR_ARG   # v != 1 for GPipe FIFO
    assert ev(B.ONEF1B, 0, 8, 1) == B.PP_ERR_ARG    # P < 1
    assert ev(B.ONEF1B, 4, 0, 1) == B.PP_ERR_ARG    # M < 1
    assert ev(B.ONEF1B, 4, 8, 2) == B.PP_ERR_ARG    # v != 1 for 1F1B
    assert ev(B.INTERLEAVED, 4, 8, 1) == B.PP_ERR_ARG  # v < 2 for interleaved
    assert ev(B.INTERLEAVED, 4, 6, 2) == B.PP_ERR_DIVISIBILITY
    assert ev(B.ONEF1B, 17, 8, 1) == B.PP_ERR_SIZE  # P beyond the limit
    assert ev(B.INTERLEAVED, 16, 32, 8) == B.PP_ERR_SIZE  # S = 128
    assert ev(B.ONEF1B, 4, 8, 1, n=-1) == B.PP_ERR_ARG
    assert ev(B.ONEF1B, 4, 8, 1, f=0) == B.PP_ERR_ARG   # NULL costs with n > 0
    assert ev(B.ONEF1B, 4, 8, 1, si=-1) == B.PP_ERR_ARG
    h = ctypes.c_void_p()
    assert L.pp_sched_plan(B.GPIPE, 4, 8, 2, ctypes.byref(h), nul) == B.PP_ERR_ARG
    assert L.pp_sched_plan(B.ONEF1B, 4, 8, 1, None, nul) == B.PP_ERR_ARG
    # partition search argument checks
    def ps(L_, P, M, n=10, ptr=8):
        return L.pp_sched_partition_search(ptr, ptr, ptr, L_, P, M, 0, 0, 0, 0, n, ptr, nul, nul,
                                           nul, nul)
    assert ps(80, 0, 8) == B.PP_ERR_ARG
    assert ps(4, 8, 8) == B.PP_ERR_ARG          # fewer layers than stages
    assert ps(300, 8, 8) == B.PP_ERR_SIZE       # L beyond 256
    assert ps(80, 8, 8, n=1 << 32) == B.PP_ERR_SIZE
    assert ps(80, 8, 8, ptr=12) == B.PP_ERR_ARG  # best_idx not 8-byte aligned
    for c in range(7):
        assert L.pp_sched_status_str(c)


def test_one_past_each_limit_is_refused_without_gpu():
    """One step past each declared limit answers PP_ERR_SIZE before any CUDA
    call (the shapes at the limits themselves run in test_gpu_limits.py)."""
    from pipeline_schedule_simulation_gb300 import binding as B
    L = B.LIB
    nul = None

    def ev(pol, P, M, v):
        return L.pp_sched_eval(pol, P, M, v, 8, 8, 1, 0, 0, nul, 0, 0, 4, nul, nul, nul, nul,
                               nul, nul, nul, 0, 0, nul, nul)
    assert ev(B.ONEF1B, 16, 32769, 1) == B.PP_ERR_SIZE       # M*v = PP_MAX_MV + 1
    assert ev(B.GPIPE, 16, 32769, 1) == B.PP_ERR_SIZE
    assert ev(B.INTERLEAVED, 2, 16386, 2) == B.PP_ERR_SIZE   # M*v = 32,772
    assert ev(B.INTERLEAVED, 13, 13, 5) == B.PP_ERR_SIZE     # P*v = 65
    assert L.pp_sched_eval_zb(B.ZB1P, 16, 32769, 8, 8, 8, 1, 0, 0, nul, 0, 0, 4, nul, nul, nul, nul, nul,
                              nul, nul, 0, 0, nul, nul) == B.PP_ERR_SIZE
    assert L.pp_sched_eval_zb(B.ZB2P, 17, 8, 8, 8, 8, 1, 0, 0, nul, 0, 0, 4, nul, nul, nul, nul, nul,
                              nul, nul, 0, 0, nul, nul) == B.PP_ERR_SIZE

    def dp(P, M, m_a, n=4, f=8, si=1):
        return L.pp_sched_eval_dualpipe(P, M, m_a, f, f, si, 0, 0, nul, 0, 0, n, nul, nul, nul, nul, nul,
                                        nul, nul, 0, 0, nul, nul)
    assert dp(0, 8, 4) == B.PP_ERR_ARG             # P < 1
    assert dp(4, 0, 0) == B.PP_ERR_ARG             # M < 1
    assert dp(4, 8, 9) == B.PP_ERR_ARG             # route A larger than M
    assert dp(4, 8, -1) == B.PP_ERR_ARG
    assert dp(4, 8, 4, n=-1) == B.PP_ERR_ARG
    assert dp(4, 8, 4, f=0) == B.PP_ERR_ARG        # NULL costs with n > 0
    assert dp(4, 8, 4, si=-1) == B.PP_ERR_ARG
    assert dp(17, 8, 4) == B.PP_ERR_SIZE
    assert dp(16, 32769, 4) == B.PP_ERR_SIZE

    def ps(L_, P, M):
        return L.pp_sched_partition_search(8, 8, 8, L_, P, M, 0, 0, 0, 0, 10, 8, 8, 8, nul, nul)

    def pr(L_, P, M, begin, n):
        return L.pp_sched_partition_search_ranks(8, 8, 8, L_, P, M, 0, 0, begin, n, 8, 8, 8, nul, nul)

    def pi(L_, P, v, M):
        return L.pp_sched_partition_search_interleaved(8, 8, 8, L_, P, v, M, 0, 0, 0, 0, 10, 8, 8, 8, nul, nul)
    assert ps(132, 16, 8) == B.PP_ERR_SIZE         # C(131, 15) does not fit 64 bits
    assert ps(257, 2, 8) == B.PP_ERR_SIZE
    assert ps(131, 16, 32769) == B.PP_ERR_SIZE     # M beyond PP_MAX_MV
    assert pr(132, 16, 8, 0, 10) == B.PP_ERR_SIZE
    assert pr(20, 4, 8, 969 - 5, 6) == B.PP_ERR_ARG   # past the last rank, C(19, 3) = 969
    assert pi(85, 16, 4, 16) == B.PP_ERR_SIZE      # C(84, 63) does not fit 64 bits
    assert pi(84, 16, 4, 8208) == B.PP_ERR_SIZE    # M*v = 32,832


def test_many_argument_errors_without_gpu():
    """pp_sched_many_*: argument errors are answered before any CUDA call."""
    from pipeline_schedule_simulation_gb300 import binding as B
    L = B.LIB
    h = ctypes.c_void_p()

    def prob(policy=B.ONEF1B, P=4, M=8, v=1, n=4, f=8, si=1):
        return B.Problem(policy, P, M, v, f, f, si, 0, 0, None, 0, 0, n, None, None, None, None, None, None)

    def prep(probs, n=None, handle=True):
        arr = (B.Problem * max(len(probs), 1))(*probs)
        return L.pp_sched_many_prepare(ctypes.cast(arr, ctypes.c_void_p), len(probs) if n is None else n,
                                       ctypes.byref(h) if handle else None, None)
    assert prep([prob()], handle=False) == B.PP_ERR_ARG
    assert prep([prob()], n=-1) == B.PP_ERR_ARG
    assert L.pp_sched_many_prepare(None, 3, ctypes.byref(h), None) == B.PP_ERR_ARG
    assert prep([prob(), prob(P=0)]) == B.PP_ERR_ARG          # the second problem's P < 1
    assert prep([prob(P=17)]) == B.PP_ERR_SIZE
    assert prep([prob(policy=B.INTERLEAVED, P=4, M=6, v=2)]) == B.PP_ERR_DIVISIBILITY
    assert prep([prob(f=0)]) == B.PP_ERR_ARG                  # NULL costs with n > 0
    assert prep([prob(si=-1)]) == B.PP_ERR_ARG
    assert prep([prob(policy=B.ZB1P)]) == B.PP_ERR_ARG        # Zero Bubble has its own entry point
    assert not h.value                                        # no handle after an error
    assert L.pp_sched_many_eval(None, None) == B.PP_ERR_ARG
    assert L.pp_sched_many_info(None, None, None, None) == B.PP_ERR_ARG
    L.pp_sched_many_destroy(None)
    # the structure's layout: pointers and 64-bit fields on their natural boundaries
    assert ctypes.sizeof(B.Problem) == 16 + 2 * 8 + 3 * 8 + 8 + 2 * 8 + 8 + 6 * 8
