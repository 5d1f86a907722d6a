"""CPU oracle for the pipeline-schedule evaluator -- TEST INFRASTRUCTURE ONLY.

A plain discrete-event simulator (``ppsim_oracle.c``, plain C99) of GPipe,
synchronous 1F1B and interleaved 1F1B, with an independent longest-path
cross-check, the pages' validity checks, a brute-force enumerator for tiny
shapes and the seeded candidate-partition scorer.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
package.  It shares no code with the CUDA library and never imports it.

Parity status of each function is stated in its docstring; every function here
is pinned by the non-GPU tests against values the pages print, closed forms, or
brute force (see ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ppsim_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libppsim_oracle.so")

GPIPE, ONEF1B, INTERLEAVED, ZB1P, ZB2P, GPIPE_FIFO = 0, 1, 2, 3, 4, 5
POLICIES = {"gpipe": GPIPE, "1f1b": ONEF1B, "interleaved": INTERLEAVED, "zb1p": ZB1P, "zb2p": ZB2P,
            "gpipe_fifo": GPIPE_FIFO}
F, B, W = 0, 1, 2

OK, ERR_ARG, ERR_DIVISIBILITY, ERR_DEADLOCK, ERR_INVARIANT, ERR_NOMEM = 0, 1, 2, 5, 6, 7
ST_OK, ST_NEG_COST, ST_OVERFLOW, ST_ZERO_COST = 0, 1, 2, 3

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    def __init__(self, code, what=""):
        super().__init__(f"oracle error {code} {what}")
        self.code = code


def build(out_path: str = _LIB_PATH, defines=()) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    src_mtime = os.path.getmtime(_SRC)
    if os.path.exists(out_path) and os.path.getmtime(out_path) >= src_mtime and not defines:
        return out_path
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-Wall", "-shared", "-fPIC", "-pthread"]
    cmd += [f"-D{d}" for d in defines]
    cmd += ["-o", tmp, _SRC]
    subprocess.check_call(cmd)
    os.replace(tmp, out_path)
    return out_path


def _bind(lib):
    i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
    i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
    c_int, c_i64, c_u64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
    lib.orc_order.argtypes = [c_int, c_int, c_int, c_int, c_int, vp, vp, vp]
    lib.orc_order.restype = c_int
    lib.orc_eval_explicit.argtypes = [c_int, c_int, c_int, vp, vp, vp, vp, vp, vp, c_int,
                                      vp, vp, vp, vp, vp, vp, vp]
    lib.orc_eval_explicit.restype = c_int
    lib.orc_eval_batch.argtypes = [c_int, c_int, c_int, c_int, c_i64, vp, vp, c_i64, c_i64, c_i64,
                                   vp, c_i64, c_i64, vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int]
    lib.orc_eval_batch.restype = c_int
    lib.orc_eval_batch_fb.argtypes = [c_int, c_int, c_int, c_int, c_i64, vp, vp, c_i64, c_i64, c_i64,
                                      vp, vp, c_i64, c_i64, vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int]
    lib.orc_eval_batch_fb.restype = c_int
    lib.orc_eval_explicit_fb.argtypes = [c_int, c_int, c_int, vp, vp, vp, vp, vp, vp, vp, c_int,
                                         vp, vp, vp, vp, vp, vp, vp]
    lib.orc_eval_explicit_fb.restype = c_int
    lib.orc_bruteforce.argtypes = [c_int, c_int, vp]
    lib.orc_bruteforce.restype = c_int
    lib.orc_search.argtypes = [vp, vp, vp, c_int, c_int, c_int, ctypes.c_int32, c_i64, c_u64,
                               c_i64, c_i64, vp, vp, vp, vp, c_int]
    lib.orc_search.restype = c_int
    lib.orc_search_ranks.argtypes = [vp, vp, vp, c_int, c_int, c_int, ctypes.c_int32, c_i64,
                                     c_i64, c_i64, vp, vp, vp, vp, c_int]
    lib.orc_search_ranks.restype = c_int
    lib.orc_search_interleaved.argtypes = [vp, vp, vp, c_int, c_int, c_int, c_int, ctypes.c_int32, c_i64, c_u64,
                                           c_i64, c_i64, vp, vp, vp, vp, c_int]
    lib.orc_search_interleaved.restype = c_int
    lib.orc_rank_split.argtypes = [c_u64, c_int, c_int, vp]
    lib.orc_rank_split.restype = None
    lib.orc_candidate_split.argtypes = [c_u64, c_i64, c_int, c_int, vp]
    lib.orc_candidate_split.restype = None
    lib.orc_binom.argtypes = [c_int, c_int]
    lib.orc_binom.restype = c_u64
    lib.orc_splitmix64.argtypes = [c_u64]
    lib.orc_splitmix64.restype = c_u64
    lib.orc_zb_inst.argtypes = [c_int, c_int, c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.orc_zb_inst.restype = c_int
    lib.orc_zb_batch.argtypes = [c_int, c_int, c_int, c_i64, vp, vp, vp, c_i64, c_i64, c_i64,
                                 vp, c_i64, c_i64, vp, vp, vp, vp, vp, vp, vp, vp, c_int]
    lib.orc_zb_batch.restype = c_int
    lib.orc_dp_inst.argtypes = [c_int, c_int, c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.orc_dp_inst.restype = c_int
    lib.orc_dp_batch.argtypes = [c_int, c_int, c_int, c_i64, vp, vp, c_i64, c_i64, c_i64,
                                 vp, c_i64, c_i64, vp, vp, vp, vp, vp, vp, vp, vp, c_int]
    lib.orc_dp_batch.restype = c_int
    del i32p, i64p
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _policy(p):
    return POLICIES[p] if isinstance(p, str) else int(p)


def order(policy, P, M, v=1, lib=None):
    """Per-device op order: (kind, chunk, mb) int32 arrays of shape [P][2Mv]."""
    lib = lib or load()
    O = 2 * M * v
    kind = np.zeros((P, O), np.int32)
    chunk = np.zeros((P, O), np.int32)
    mb = np.zeros((P, O), np.int32)
    for k in range(P):
        n = lib.orc_order(_policy(policy), P, M, v, k, _ptr(kind[k]), _ptr(chunk[k]), _ptr(mb[k]))
        if n < 0:
            raise OracleError(-n, f"order({policy},{P},{M},{v})")
    return kind, chunk, mb


def eval_explicit(P, M, v, kind, chunk, mb, tf, tb, comm=None, method=2, lib=None, comm_b=None):
    """Evaluate one instance with an explicit order.

    tf, tb: [S][M] costs; comm: [S-1] or None; comm_b: [S-1] latency of the
    backward edges (None: the same as comm).  method 0 = event simulation,
    1 = longest path, 2 = both (must agree).  Returns a dict with start, end
    ([P][O]), makespan, busy, idle, bub (num, den), peak; raises OracleError on
    deadlock or a failed validity check.
    """
    lib = lib or load()
    S, O = P * v, 2 * M * v
    kind = np.ascontiguousarray(kind, np.int32)
    chunk = np.ascontiguousarray(chunk, np.int32)
    mb = np.ascontiguousarray(mb, np.int32)
    tf = np.ascontiguousarray(np.broadcast_to(np.asarray(tf, np.int64), (S, M)))
    tb = np.ascontiguousarray(np.broadcast_to(np.asarray(tb, np.int64), (S, M)))
    cm = None if comm is None else np.ascontiguousarray(np.broadcast_to(np.asarray(comm, np.int64), (max(S - 1, 1),)))
    cmb = None if comm_b is None else np.ascontiguousarray(
        np.broadcast_to(np.asarray(comm_b, np.int64), (max(S - 1, 1),)))
    start = np.zeros((P, O), np.int64)
    end = np.zeros((P, O), np.int64)
    mk = np.zeros(1, np.int64)
    busy = np.zeros(P, np.int64)
    idle = np.zeros(P, np.int64)
    bub = np.zeros(2, np.int64)
    peak = np.zeros(P, np.int32)
    rc = lib.orc_eval_explicit_fb(P, M, v, _ptr(kind), _ptr(chunk), _ptr(mb), _ptr(tf), _ptr(tb),
                                  _ptr(cm), _ptr(cmb), method, _ptr(start), _ptr(end), _ptr(mk), _ptr(busy),
                                  _ptr(idle), _ptr(bub), _ptr(peak))
    if rc != OK:
        raise OracleError(rc, "eval_explicit")
    return dict(start=start, end=end, makespan=int(mk[0]), busy=busy, idle=idle,
                bub=(int(bub[0]), int(bub[1])), peak=peak)


def evaluate(policy, P, M, v, tf, tb, comm=None, method=2, lib=None, comm_b=None):
    """Generate the policy's order and evaluate one instance (see eval_explicit)."""
    kind, chunk, mb = order(policy, P, M, v, lib=lib)
    r = eval_explicit(P, M, v, kind, chunk, mb, tf, tb, comm, method, lib=lib, comm_b=comm_b)
    r.update(kind=kind, chunk=chunk, mb=mb)
    return r


def eval_batch(policy, P, M, v, cost_f, cost_b, strides, comm=None, comm_strides=(0, 0), n=None,
               op_times=False, method=0, nthreads=1, lib=None, comm_b=None):
    """Evaluate n instances.  cost_f/cost_b are flat int32 buffers indexed by
    element strides (inst, stage, mb); comm a flat int32 buffer indexed by
    (inst, boundary) strides or None; comm_b the backward edges' latency with
    comm's strides (None: the same as comm).  Returns dict of numpy outputs."""
    lib = lib or load()
    S, O = P * v, 2 * M * v
    cost_f = np.ascontiguousarray(cost_f, np.int32).reshape(-1)
    cost_b = np.ascontiguousarray(cost_b, np.int32).reshape(-1)
    cm = None if comm is None else np.ascontiguousarray(comm, np.int32).reshape(-1)
    cmb = None if comm_b is None else np.ascontiguousarray(comm_b, np.int32).reshape(-1)
    if n is None:
        raise ValueError("n required")
    out = dict(
        makespan=np.zeros(n, np.int64), idle=np.zeros((n, P), np.int64),
        bub_num=np.zeros(n, np.int64), bub_den=np.zeros(n, np.int64),
        peak=np.zeros(P, np.int32), status=np.zeros(n, np.int8))
    if op_times:
        out["op_start"] = np.zeros((n, P, O), np.int64)
        out["op_end"] = np.zeros((n, P, O), np.int64)
    rc = lib.orc_eval_batch_fb(_policy(policy), P, M, v, n, _ptr(cost_f), _ptr(cost_b),
                               strides[0], strides[1], strides[2], _ptr(cm), _ptr(cmb), comm_strides[0],
                               comm_strides[1], _ptr(out["makespan"]), _ptr(out["idle"]),
                            _ptr(out["bub_num"]), _ptr(out["bub_den"]), _ptr(out["peak"]),
                            _ptr(out["status"]), _ptr(out.get("op_start")), _ptr(out.get("op_end")),
                            method, nthreads)
    if rc != OK:
        raise OracleError(rc, "eval_batch")
    return out


def bruteforce(P, M, lib=None):
    """Exhaustive check over every valid order for tiny P, M (unit costs):
    returns dict(valid, deadlocked, min_makespan, n_optimal, min_peak0, min_peakmax)."""
    lib = lib or load()
    out = np.zeros(6, np.int64)
    rc = lib.orc_bruteforce(P, M, _ptr(out))
    if rc != OK:
        raise OracleError(rc, "bruteforce")
    keys = ["valid", "deadlocked", "min_makespan", "n_optimal", "min_peak0", "min_peakmax"]
    return dict(zip(keys, (int(x) for x in out)))


def candidate_split(seed, c, L, P, lib=None):
    """First layer of each stage for candidate c (length P+1, last = L)."""
    lib = lib or load()
    first = np.zeros(P + 1, np.int32)
    lib.orc_candidate_split(ctypes.c_uint64(seed & (2**64 - 1)), c, L, P, _ptr(first))
    return first


def search(layer_tf, layer_tb, layer_act, P, M, comm, cap, seed, c_lo, c_hi, nthreads=1, lib=None):
    """Score candidates [c_lo, c_hi) under 1F1B; returns dict(all_makespan,
    best_idx, best_makespan, first) -- see orc_search."""
    lib = lib or load()
    ltf = np.ascontiguousarray(layer_tf, np.int32)
    ltb = np.ascontiguousarray(layer_tb, np.int32)
    lact = np.ascontiguousarray(layer_act, np.int64)
    L = ltf.shape[0]
    all_mk = np.zeros(c_hi - c_lo, np.int32)
    bi = np.zeros(1, np.int64)
    bm = np.zeros(1, np.int64)
    first = np.zeros(P + 1, np.int32)
    rc = lib.orc_search(_ptr(ltf), _ptr(ltb), _ptr(lact), L, P, M, comm, cap,
                        ctypes.c_uint64(seed & (2**64 - 1)), c_lo, c_hi, _ptr(all_mk),
                        _ptr(bi), _ptr(bm), _ptr(first), nthreads)
    if rc != OK:
        raise OracleError(rc, "search")
    return dict(all_makespan=all_mk, best_idx=int(bi[0]), best_makespan=int(bm[0]), first=first)


def search_ranks(layer_tf, layer_tb, layer_act, P, M, comm, cap, r_lo, r_hi, nthreads=1, lib=None):
    """Exhaustive search over the splits of colex ranks [r_lo, r_hi); returns
    dict(all_makespan, best_idx (a rank), best_makespan, first) -- see
    orc_search_ranks."""
    lib = lib or load()
    ltf = np.ascontiguousarray(layer_tf, np.int32)
    ltb = np.ascontiguousarray(layer_tb, np.int32)
    lact = np.ascontiguousarray(layer_act, np.int64)
    L = ltf.shape[0]
    all_mk = np.zeros(r_hi - r_lo, np.int32)
    bi = np.zeros(1, np.int64)
    bm = np.zeros(1, np.int64)
    first = np.zeros(P + 1, np.int32)
    rc = lib.orc_search_ranks(_ptr(ltf), _ptr(ltb), _ptr(lact), L, P, M, comm, cap, r_lo, r_hi, _ptr(all_mk),
                              _ptr(bi), _ptr(bm), _ptr(first), nthreads)
    if rc != OK:
        raise OracleError(rc, "search_ranks")
    return dict(all_makespan=all_mk, best_idx=int(bi[0]), best_makespan=int(bm[0]), first=first)


def search_interleaved(layer_tf, layer_tb, layer_act, P, v, M, comm, cap, seed, c_lo, c_hi, nthreads=1, lib=None):
    """Seeded search over interleaved layouts (S = P*v contiguous ranges);
    returns dict(all_makespan, best_idx, best_makespan, first [S+1]) -- see
    orc_search_interleaved."""
    lib = lib or load()
    ltf = np.ascontiguousarray(layer_tf, np.int32)
    ltb = np.ascontiguousarray(layer_tb, np.int32)
    lact = np.ascontiguousarray(layer_act, np.int64)
    L = ltf.shape[0]
    all_mk = np.zeros(c_hi - c_lo, np.int32)
    bi = np.zeros(1, np.int64)
    bm = np.zeros(1, np.int64)
    first = np.zeros(P * v + 1, np.int32)
    rc = lib.orc_search_interleaved(_ptr(ltf), _ptr(ltb), _ptr(lact), L, P, v, M, comm, cap,
                                    ctypes.c_uint64(seed & (2**64 - 1)), c_lo, c_hi, _ptr(all_mk),
                                    _ptr(bi), _ptr(bm), _ptr(first), nthreads)
    if rc != OK:
        raise OracleError(rc, "search_interleaved")
    return dict(all_makespan=all_mk, best_idx=int(bi[0]), best_makespan=int(bm[0]), first=first)


def rank_split(r, L, P, lib=None):
    """Stage starts [P+1] of the split of colex rank r."""
    first = np.zeros(P + 1, np.int32)
    (lib or load()).orc_rank_split(ctypes.c_uint64(r), L, P, _ptr(first))
    return first


def binom(n, k, lib=None):
    return int((lib or load()).orc_binom(n, k))


def splitmix64(state, lib=None):
    return int((lib or load()).orc_splitmix64(ctypes.c_uint64(state & (2**64 - 1))))


def zb_evaluate(policy, P, M, tf, tb, tw, comm=None, lib=None):
    """One Zero Bubble instance (ZB1P or ZB2P).

    tf, tb: [P][M] costs >= 1, tw: [P][M] costs >= 0 (scalars broadcast);
    comm: [P-1] or None.  Returns start, end ([P][3][M]: device, kind F/B/W, microbatch),
    makespan, busy, idle, bub (num, den) and peak (held microbatches, +1 at F,
    -1 at W).  Raises OracleError on a cost out of range or a failed validity
    check.
    Parity: pinned by hand-derived worked examples, the W-free reduction to
    1F1B and to the explicit-order evaluator, and an independent tick-stepped
    simulation (tests/test_oracle_pins.py)."""
    lib = lib or load()
    full = lambda a: np.ascontiguousarray(np.broadcast_to(np.asarray(a, np.int64), (P, M)))
    tf, tb, tw = full(tf), full(tb), full(tw)
    cm = None if comm is None else np.ascontiguousarray(np.broadcast_to(np.asarray(comm, np.int64), (max(P - 1, 1),)))
    start = np.zeros((P, 3, M), np.int64)
    end = np.zeros((P, 3, M), np.int64)
    mk = np.zeros(1, np.int64)
    busy = np.zeros(P, np.int64)
    idle = np.zeros(P, np.int64)
    bub = np.zeros(2, np.int64)
    peak = np.zeros(P, np.int32)
    rc = lib.orc_zb_inst(_policy(policy), P, M, _ptr(tf), _ptr(tb), _ptr(tw), _ptr(cm), _ptr(start), _ptr(end),
                         _ptr(mk), _ptr(busy), _ptr(idle), _ptr(bub), _ptr(peak))
    if rc != OK:
        raise OracleError(rc, "zb_evaluate")
    return dict(start=start, end=end, makespan=int(mk[0]), busy=busy, idle=idle,
                bub=(int(bub[0]), int(bub[1])), peak=peak)


def zb_batch(policy, P, M, cost_f, cost_b, cost_w, strides, comm=None, comm_strides=(0, 0), n=None,
             op_times=False, nthreads=1, lib=None):
    """Zero Bubble batch with the library's input conventions (int32 costs
    through element strides shared by F, B and W; comm [inst][boundary]).
    Returns makespan, idle [n][P], bub_num, bub_den, peak [n][P], status and
    optionally op_start / op_end [n][P][3][M]."""
    lib = lib or load()
    cf = np.ascontiguousarray(cost_f, np.int32)
    cb = np.ascontiguousarray(cost_b, np.int32)
    cw = np.ascontiguousarray(cost_w, np.int32)
    cm = None if comm is None else np.ascontiguousarray(comm, np.int32)
    out = dict(makespan=np.zeros(n, np.int64), idle=np.zeros((n, P), np.int64),
               bub_num=np.zeros(n, np.int64), bub_den=np.zeros(n, np.int64),
               peak=np.zeros((n, P), np.int32), status=np.zeros(n, np.int8))
    os_ = oe = None
    if op_times:
        os_ = np.zeros((n, P, 3, M), np.int64)
        oe = np.zeros((n, P, 3, M), np.int64)
    rc = lib.orc_zb_batch(_policy(policy), P, M, n, _ptr(cf), _ptr(cb), _ptr(cw), strides[0], strides[1],
                          strides[2], _ptr(cm), comm_strides[0], comm_strides[1],
                          _ptr(out["makespan"]), _ptr(out["idle"]), _ptr(out["bub_num"]), _ptr(out["bub_den"]),
                          _ptr(out["peak"]), _ptr(out["status"]), _ptr(os_), _ptr(oe), nthreads)
    if rc != OK:
        raise OracleError(rc, "zb_batch")
    if op_times:
        out["op_start"], out["op_end"] = os_, oe
    return out


def dp_evaluate(P, MA, MB, tf, tb, comm=None, lib=None):
    """One DualPipe instance: route A carries microbatches 0..MA-1 from device 0,
    route B microbatches MA..MA+MB-1 from device P-1 (see orc_dp_inst).

    tf, tb: [P blocks][M] costs >= 1 (scalars broadcast); comm: [P-1] per link
    or None.  Returns start, end ([P][2][M]: block, kind F/B, microbatch),
    makespan, busy, idle, bub (num, den) and peak per device (+1 at F, -1 at B).
    Parity: pinned by the reduction of one route to 1F1B, the mirror symmetry,
    the page's peak of p+1 and an independent tick-stepped simulation
    (tests/test_oracle_dualpipe.py)."""
    lib = lib or load()
    M = MA + MB
    full = lambda a: np.ascontiguousarray(np.broadcast_to(np.asarray(a, np.int64), (P, M)))
    tf, tb = full(tf), full(tb)
    cm = None if comm is None else np.ascontiguousarray(np.broadcast_to(np.asarray(comm, np.int64), (max(P - 1, 1),)))
    start = np.zeros((P, 2, M), np.int64)
    end = np.zeros((P, 2, M), np.int64)
    mk = np.zeros(1, np.int64)
    busy = np.zeros(P, np.int64)
    idle = np.zeros(P, np.int64)
    bub = np.zeros(2, np.int64)
    peak = np.zeros(P, np.int32)
    rc = lib.orc_dp_inst(P, MA, MB, _ptr(tf), _ptr(tb), _ptr(cm), _ptr(start), _ptr(end), _ptr(mk), _ptr(busy),
                         _ptr(idle), _ptr(bub), _ptr(peak))
    if rc != OK:
        raise OracleError(rc, "dp_evaluate")
    return dict(start=start, end=end, makespan=int(mk[0]), busy=busy, idle=idle,
                bub=(int(bub[0]), int(bub[1])), peak=peak)


def dp_batch(P, MA, MB, cost_f, cost_b, strides, comm=None, comm_strides=(0, 0), n=None, op_times=False,
             nthreads=1, lib=None):
    """DualPipe batch with the library's input conventions (int32 costs
    [inst][block][microbatch] through element strides; comm [inst][link]).
    Returns makespan, idle [n][P], bub_num, bub_den, peak [n][P], status and
    optionally op_start / op_end [n][P][2][M]."""
    lib = lib or load()
    M = MA + MB
    cf = np.ascontiguousarray(cost_f, np.int32)
    cb = np.ascontiguousarray(cost_b, np.int32)
    cm = None if comm is None else np.ascontiguousarray(comm, np.int32)
    out = dict(makespan=np.zeros(n, np.int64), idle=np.zeros((n, P), np.int64),
               bub_num=np.zeros(n, np.int64), bub_den=np.zeros(n, np.int64),
               peak=np.zeros((n, P), np.int32), status=np.zeros(n, np.int8))
    os_ = oe = None
    if op_times:
        os_ = np.zeros((n, P, 2, M), np.int64)
        oe = np.zeros((n, P, 2, M), np.int64)
    rc = lib.orc_dp_batch(P, MA, MB, n, _ptr(cf), _ptr(cb), strides[0], strides[1], strides[2], _ptr(cm),
                          comm_strides[0], comm_strides[1], _ptr(out["makespan"]), _ptr(out["idle"]),
                          _ptr(out["bub_num"]), _ptr(out["bub_den"]), _ptr(out["peak"]), _ptr(out["status"]),
                          _ptr(os_), _ptr(oe), nthreads)
    if rc != OK:
        raise OracleError(rc, "dp_batch")
    if op_times:
        out["op_start"], out["op_end"] = os_, oe
    return out
