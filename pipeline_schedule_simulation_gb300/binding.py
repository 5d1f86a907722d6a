"""ctypes binding of libppsched (include/ppsched.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  PyTorch
provides device memory and streams.  There is no CPU fallback: if the library
has not been built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build_lib

GPIPE, ONEF1B, INTERLEAVED, ZB1P, ZB2P, GPIPE_FIFO = 0, 1, 2, 3, 4, 5
POLICIES = {"gpipe": GPIPE, "1f1b": ONEF1B, "interleaved": INTERLEAVED, "zb1p": ZB1P, "zb2p": ZB2P,
            "gpipe_fifo": GPIPE_FIFO}

PP_OK, PP_ERR_ARG, PP_ERR_DIVISIBILITY, PP_ERR_SIZE, PP_ERR_CUDA, PP_ERR_DEADLOCK, PP_ERR_INTERNAL = range(7)
ST_OK, ST_NEG_COST, ST_OVERFLOW, ST_ZERO_COST = 0, 1, 2, 3

EXPORTS = ("pp_sched_plan", "pp_sched_plan_info", "pp_sched_plan_ops", "pp_sched_plan_destroy",
           "pp_sched_eval", "pp_sched_partition_search", "pp_sched_status_str",
           "pp_sched_cache_clear", "pp_sched_eval_noalloc", "pp_sched_eval_zb",
           "pp_sched_partition_search_ranks", "pp_sched_partition_search_interleaved", "pp_sched_eval_fb",
           "pp_sched_eval_host", "pp_sched_eval_host_workspace", "pp_sched_many_prepare", "pp_sched_many_eval",
           "pp_sched_many_info", "pp_sched_many_destroy", "pp_sched_eval_dualpipe")


class Problem(ctypes.Structure):
    """pp_problem_t: one problem of pp_sched_many_* (the arguments of
    pp_sched_eval without per-op output)."""
    _fields_ = [("policy", ctypes.c_int), ("P", ctypes.c_int), ("M", ctypes.c_int), ("v", ctypes.c_int),
                ("cost_f", ctypes.c_void_p), ("cost_b", ctypes.c_void_p),
                ("stride_inst", ctypes.c_int64), ("stride_stage", ctypes.c_int64), ("stride_mb", ctypes.c_int64),
                ("comm", ctypes.c_void_p), ("comm_stride_inst", ctypes.c_int64), ("comm_stride_bnd", ctypes.c_int64),
                ("n_instances", ctypes.c_int64), ("makespan", ctypes.c_void_p), ("idle", ctypes.c_void_p),
                ("bub_num", ctypes.c_void_p), ("bub_den", ctypes.c_void_p), ("peak", ctypes.c_void_p),
                ("status", ctypes.c_void_p)]


class PPSchedError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_str(code)} (code {code})")


def _load():
    path = build_lib.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"libppsched.so is not built ({path}); run __graft_entry__.build() or "
            "python -m pipeline_schedule_simulation_gb300.build_lib")
    lib = ctypes.CDLL(path)
    vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
    lib.pp_sched_plan.argtypes = [i32, i32, i32, i32, ctypes.POINTER(vp), vp]
    lib.pp_sched_plan.restype = i32
    lib.pp_sched_plan_info.argtypes = [vp, vp]
    lib.pp_sched_plan_info.restype = i32
    lib.pp_sched_plan_ops.argtypes = [vp, vp, vp, vp]
    lib.pp_sched_plan_ops.restype = i32
    lib.pp_sched_plan_destroy.argtypes = [vp]
    lib.pp_sched_plan_destroy.restype = None
    lib.pp_sched_eval.argtypes = [i32, i32, i32, i32, vp, vp, i64, i64, i64, vp, i64, i64, i64,
                                  vp, vp, vp, vp, vp, vp, vp, i64, i64, vp, vp]
    lib.pp_sched_eval.restype = i32
    lib.pp_sched_many_prepare.argtypes = [vp, i32, ctypes.POINTER(vp), vp]
    lib.pp_sched_many_prepare.restype = i32
    lib.pp_sched_many_eval.argtypes = [vp, vp]
    lib.pp_sched_many_eval.restype = i32
    lib.pp_sched_many_info.argtypes = [vp, vp, vp, vp]
    lib.pp_sched_many_info.restype = i32
    lib.pp_sched_many_destroy.argtypes = [vp]
    lib.pp_sched_many_destroy.restype = None
    lib.pp_sched_eval_fb.argtypes = [i32, i32, i32, i32, vp, vp, i64, i64, i64, vp, vp, i64, i64, i64,
                                     vp, vp, vp, vp, vp, vp, vp, i64, i64, vp, vp]
    lib.pp_sched_eval_fb.restype = i32
    lib.pp_sched_partition_search.argtypes = [vp, vp, vp, i32, i32, i32, ctypes.c_int32, i64, u64,
                                              i64, i64, vp, vp, vp, vp, vp]
    lib.pp_sched_partition_search.restype = i32
    lib.pp_sched_partition_search_ranks.argtypes = [vp, vp, vp, i32, i32, i32, ctypes.c_int32, i64, i64, i64,
                                                    vp, vp, vp, vp, vp]
    lib.pp_sched_partition_search_ranks.restype = i32
    lib.pp_sched_partition_search_interleaved.argtypes = [vp, vp, vp, i32, i32, i32, i32, ctypes.c_int32, i64, u64,
                                                          i64, i64, vp, vp, vp, vp, vp]
    lib.pp_sched_partition_search_interleaved.restype = i32
    lib.pp_sched_status_str.argtypes = [i32]
    lib.pp_sched_status_str.restype = ctypes.c_char_p
    lib.pp_sched_eval_noalloc.argtypes = [i32, i32, i32, vp, vp, i64, i64, i64, vp, i64, i64, i64,
                                          vp, vp, vp, vp, vp, vp, vp]
    lib.pp_sched_eval_noalloc.restype = i32
    lib.pp_sched_eval_zb.argtypes = [i32, i32, i32, vp, vp, vp, i64, i64, i64, vp, i64, i64, i64,
                                     vp, vp, vp, vp, vp, vp, vp, i64, i64, vp, vp]
    lib.pp_sched_eval_zb.restype = i32
    lib.pp_sched_eval_dualpipe.argtypes = [i32, i32, i32, vp, vp, i64, i64, i64, vp, i64, i64, i64,
                                           vp, vp, vp, vp, vp, vp, vp, i64, i64, vp, vp]
    lib.pp_sched_eval_dualpipe.restype = i32
    lib.pp_sched_eval_host.argtypes = [i32, i32, i32, i32, vp, vp, vp, i64, vp, ctypes.c_size_t,
                                       vp, vp, vp, vp, vp, vp, vp]
    lib.pp_sched_eval_host.restype = i32
    lib.pp_sched_eval_host_workspace.argtypes = [i32, i32, i32, i64]
    lib.pp_sched_eval_host_workspace.restype = ctypes.c_size_t
    lib.pp_sched_cache_clear.argtypes = []
    lib.pp_sched_cache_clear.restype = None
    return lib


LIB = _load()


def status_str(code: int) -> str:
    return LIB.pp_sched_status_str(code).decode()


def _check(rc: int, where: str):
    if rc != PP_OK:
        raise PPSchedError(rc, where)


def _policy(p) -> int:
    return POLICIES[p] if isinstance(p, str) else int(p)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """A library-owned plan (pp_sched_plan); freed when garbage-collected."""

    def __init__(self, policy, P, M, v=1, stream=None):
        self._h = ctypes.c_void_p()
        _check(LIB.pp_sched_plan(_policy(policy), P, M, v, ctypes.byref(self._h), _stream(stream)),
               "pp_sched_plan")
        info = (ctypes.c_int32 * 8)()
        _check(LIB.pp_sched_plan_info(self._h, info), "pp_sched_plan_info")
        self.rounds, self.ops_per_device, self.value_slots, self.register_path = info[0:4]
        self.P, self.M, self.v, self.policy = info[4:8]

    def tables(self):
        """Host copies: (ops uint32 [P][O], peak int32 [P], round int32 [P][O])."""
        O = self.ops_per_device
        ops = torch.zeros(self.P * O, dtype=torch.int64)
        buf = (ctypes.c_uint32 * (self.P * O))()
        peak = (ctypes.c_int32 * self.P)()
        rnd = (ctypes.c_int32 * (self.P * O))()
        _check(LIB.pp_sched_plan_ops(self._h, buf, peak, rnd), "pp_sched_plan_ops")
        ops = torch.tensor(list(buf), dtype=torch.int64).reshape(self.P, O)
        return ops, torch.tensor(list(peak), dtype=torch.int32), \
            torch.tensor(list(rnd), dtype=torch.int32).reshape(self.P, O)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            LIB.pp_sched_plan_destroy(h)
            self._h = None


def op_fields(ops):
    """Split packed ops (PP_OP_* layout) into (kind, chunk, microbatch)."""
    ops = ops.to(torch.int64)
    return (ops >> 31) & 1, (ops >> 24) & 0x7F, ops & 0xFFFFFF


def evaluate(policy, P, M, v, cost_f, cost_b, strides, n, comm=None, comm_strides=(0, 0),
             outputs=("makespan", "idle", "bub_num", "bub_den", "peak", "status"),
             op_times=False, op_strides=None, out=None, stream=None, comm_b=None):
    """Call pp_sched_eval (pp_sched_eval_fb when comm_b, the backward edges'
    latency with comm's strides, is given) on DEVICE tensors.

    cost_f / cost_b / comm are int32 CUDA tensors addressed through element
    strides (see the header).  Returns a dict of int32/int64/int8 CUDA tensors;
    `out` may supply preallocated ones.  op_times adds op_start / op_end
    [n][P][O] (or through op_strides = (inst, op))."""
    pol = _policy(policy)
    dev = cost_f.device
    out = dict(out or {})
    O = 2 * M * v

    def want(name, shape, dtype):
        if name in out:
            return out[name]
        t = torch.empty(shape, dtype=dtype, device=dev)
        out[name] = t
        return t

    mk = want("makespan", (n,), torch.int32) if "makespan" in outputs else None
    idle = want("idle", (n, P), torch.int32) if "idle" in outputs else None
    bn = want("bub_num", (n,), torch.int64) if "bub_num" in outputs else None
    bd = want("bub_den", (n,), torch.int64) if "bub_den" in outputs else None
    pk = want("peak", (P,), torch.int32) if "peak" in outputs else None
    stt = want("status", (n,), torch.int8) if "status" in outputs else None
    os_ = oe = None
    if op_times:
        os_ = want("op_start", (n, P, O), torch.int32)
        oe = want("op_end", (n, P, O), torch.int32)
        if op_strides is None:
            op_strides = (P * O, 1)
    else:
        op_strides = (0, 0)
    if comm_b is not None:
        rc = LIB.pp_sched_eval_fb(pol, P, M, v, _ptr(cost_f), _ptr(cost_b), strides[0], strides[1], strides[2],
                                  _ptr(comm), _ptr(comm_b), comm_strides[0], comm_strides[1], n,
                                  _ptr(mk), _ptr(idle), _ptr(bn), _ptr(bd), _ptr(pk), _ptr(os_), _ptr(oe),
                                  op_strides[0], op_strides[1], _ptr(stt), _stream(stream))
        _check(rc, "pp_sched_eval_fb")
        return out
    rc = LIB.pp_sched_eval(pol, P, M, v, _ptr(cost_f), _ptr(cost_b), strides[0], strides[1], strides[2],
                           _ptr(comm), comm_strides[0], comm_strides[1], n,
                           _ptr(mk), _ptr(idle), _ptr(bn), _ptr(bd), _ptr(pk), _ptr(os_), _ptr(oe),
                           op_strides[0], op_strides[1], _ptr(stt), _stream(stream))
    _check(rc, "pp_sched_eval")
    return out


def evaluate_dualpipe(P, M, m_a, cost_f, cost_b, strides, n, comm=None, comm_strides=(0, 0),
                      outputs=("makespan", "idle", "bub_num", "bub_den", "peak", "status"),
                      op_times=False, op_strides=None, out=None, stream=None):
    """Call pp_sched_eval_dualpipe on DEVICE tensors: microbatches 0..m_a-1
    enter at device 0, m_a..M-1 at device P-1.

    cost_f / cost_b are indexed (instance, block, microbatch) through the
    element strides; comm (instance, link).  Returns a dict of CUDA tensors;
    `peak` is per instance [n][P].  op_times adds op_start / op_end
    [n][P blocks][2][M] (kind 0 = F, 1 = B), or through op_strides = (inst, op)."""
    dev = cost_f.device
    out = dict(out or {})

    def want(name, shape, dtype):
        if name in out:
            return out[name]
        t = torch.empty(shape, dtype=dtype, device=dev)
        out[name] = t
        return t

    mk = want("makespan", (n,), torch.int32) if "makespan" in outputs else None
    idle = want("idle", (n, P), torch.int32) if "idle" in outputs else None
    bn = want("bub_num", (n,), torch.int64) if "bub_num" in outputs else None
    bd = want("bub_den", (n,), torch.int64) if "bub_den" in outputs else None
    pk = want("peak", (n, P), torch.int32) if "peak" in outputs else None
    stt = want("status", (n,), torch.int8) if "status" in outputs else None
    os_ = oe = None
    if op_times:
        os_ = want("op_start", (n, P, 2, M), torch.int32)
        oe = want("op_end", (n, P, 2, M), torch.int32)
        if op_strides is None:
            op_strides = (P * 2 * M, 1)
    else:
        op_strides = (0, 0)
    rc = LIB.pp_sched_eval_dualpipe(P, M, m_a, _ptr(cost_f), _ptr(cost_b), strides[0], strides[1], strides[2],
                                    _ptr(comm), comm_strides[0], comm_strides[1], n, _ptr(mk), _ptr(idle),
                                    _ptr(bn), _ptr(bd), _ptr(pk), _ptr(os_), _ptr(oe), op_strides[0],
                                    op_strides[1], _ptr(stt), _stream(stream))
    _check(rc, "pp_sched_eval_dualpipe")
    return out


def evaluate_zb(policy, P, M, cost_f, cost_b, cost_w, strides, n, comm=None, comm_strides=(0, 0),
                outputs=("makespan", "idle", "bub_num", "bub_den", "peak", "status"),
                op_times=False, op_strides=None, out=None, stream=None):
    """Call pp_sched_eval_zb (ZB1P / ZB2P) on DEVICE tensors.

    cost_f / cost_b / cost_w share the element strides (inst, stage, mb).
    Returns a dict of CUDA tensors; `peak` is per instance [n][P].  op_times
    adds op_start / op_end [n][P][3][M] (kind 0 = F, 1 = B, 2 = W), or through
    op_strides = (inst, op)."""
    pol = _policy(policy)
    dev = cost_f.device
    out = dict(out or {})

    def want(name, shape, dtype):
        if name in out:
            return out[name]
        t = torch.empty(shape, dtype=dtype, device=dev)
        out[name] = t
        return t

    mk = want("makespan", (n,), torch.int32) if "makespan" in outputs else None
    idle = want("idle", (n, P), torch.int32) if "idle" in outputs else None
    bn = want("bub_num", (n,), torch.int64) if "bub_num" in outputs else None
    bd = want("bub_den", (n,), torch.int64) if "bub_den" in outputs else None
    pk = want("peak", (n, P), torch.int32) if "peak" in outputs else None
    stt = want("status", (n,), torch.int8) if "status" in outputs else None
    os_ = oe = None
    if op_times:
        os_ = want("op_start", (n, P, 3, M), torch.int32)
        oe = want("op_end", (n, P, 3, M), torch.int32)
        if op_strides is None:
            op_strides = (P * 3 * M, 1)
    else:
        op_strides = (0, 0)
    rc = LIB.pp_sched_eval_zb(pol, P, M, _ptr(cost_f), _ptr(cost_b), _ptr(cost_w), strides[0], strides[1],
                              strides[2], _ptr(comm), comm_strides[0], comm_strides[1], n,
                              _ptr(mk), _ptr(idle), _ptr(bn), _ptr(bd), _ptr(pk), _ptr(os_), _ptr(oe),
                              op_strides[0], op_strides[1], _ptr(stt), _stream(stream))
    _check(rc, "pp_sched_eval_zb")
    return out


class Many:
    """pp_sched_many_*: many problems, each with its own shape, evaluated
    together.  `problems` is a list of dicts with the keys policy, P, M, v,
    cost_f, cost_b, strides (inst, stage, mb), n and optionally comm,
    comm_strides, and `out` (a dict of preallocated CUDA output tensors:
    makespan, idle, bub_num, bub_den, peak, status; missing ones are
    allocated).  The tensors are kept alive by this object; the library keeps
    their pointers, so rewrite their contents in place between evaluations.
    prepare() builds plans and tables (it may allocate and synchronize);
    __call__ enqueues one evaluation of every problem on `stream`."""

    def __init__(self, problems, stream=None):
        self.handle = None
        self.problems = []
        arr = (Problem * max(len(problems), 1))()
        for i, q in enumerate(problems):
            P, n = q["P"], q["n"]
            out = dict(q.get("out") or {})
            dev = q["cost_f"].device
            for k, shape, dt in (("makespan", (n,), torch.int32), ("idle", (n, P), torch.int32),
                                 ("bub_num", (n,), torch.int64), ("bub_den", (n,), torch.int64),
                                 ("peak", (P,), torch.int32), ("status", (n,), torch.int8)):
                if k not in out:
                    out[k] = torch.empty(shape, dtype=dt, device=dev)
            comm = q.get("comm")
            cs = q.get("comm_strides", (0, 0))
            si, ss, sm = q["strides"]
            arr[i] = Problem(_policy(q["policy"]), P, q["M"], q.get("v", 1), _ptr(q["cost_f"]), _ptr(q["cost_b"]),
                             si, ss, sm, _ptr(comm), cs[0], cs[1], n, _ptr(out["makespan"]), _ptr(out["idle"]),
                             _ptr(out["bub_num"]), _ptr(out["bub_den"]), _ptr(out["peak"]), _ptr(out["status"]))
            self.problems.append(dict(q, out=out))
        h = ctypes.c_void_p()
        _check(LIB.pp_sched_many_prepare(ctypes.cast(arr, ctypes.c_void_p), len(problems), ctypes.byref(h),
                                         _stream(stream)), "pp_sched_many_prepare")
        self.handle = h

    def info(self):
        f, l_, o = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(LIB.pp_sched_many_info(self.handle, ctypes.byref(f), ctypes.byref(l_), ctypes.byref(o)),
               "pp_sched_many_info")
        return {"fused_problems": f.value, "launches": l_.value, "other_problems": o.value}

    def __call__(self, stream=None):
        _check(LIB.pp_sched_many_eval(self.handle, _stream(stream)), "pp_sched_many_eval")
        return [q["out"] for q in self.problems]

    def close(self):
        if self.handle:
            LIB.pp_sched_many_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def evaluate_host(policy, P, M, v, cost_f, cost_b, n, comm=None, stream=None, staging=None, workspace_bytes=None):
    """End-to-end call from HOST buffers through pp_sched_eval_host (the public
    entry for host-resident inputs): cost_f / cost_b are host int32 tensors in
    the instance-minor layout [S][M][n] (page-locked for asynchronous copies),
    comm [S-1][n] or None.  The library copies them to a device workspace,
    evaluates and copies the summary outputs back on `stream`.  `staging` (a
    dict) keeps the workspace and the host output tensors across calls;
    `workspace_bytes` bounds the workspace (the default holds the whole batch).
    Returns (outputs on host, bytes host->device, bytes device->host); the
    outputs are valid once the stream has completed."""
    staging = staging if staging is not None else {}
    S = P * v
    need = LIB.pp_sched_eval_host_workspace(P, M, v, n)
    want_ws = int(workspace_bytes) if workspace_bytes is not None else int(need)
    ws = staging.get("workspace")
    if ws is None or ws.numel() != want_ws:
        ws = torch.empty(max(want_ws, 1), dtype=torch.uint8, device="cuda")
        staging["workspace"] = ws
    host = {}
    shapes = {"makespan": ((n,), torch.int32), "idle": ((n, P), torch.int32), "bub_num": ((n,), torch.int64),
              "bub_den": ((n,), torch.int64), "peak": ((P,), torch.int32), "status": ((n,), torch.int8)}
    for k, (shape, dt) in shapes.items():
        hk = staging.get("host_" + k)
        if hk is None or tuple(hk.shape) != shape:
            hk = torch.empty(shape, dtype=dt, pin_memory=True)
            staging["host_" + k] = hk
        host[k] = hk
    rc = LIB.pp_sched_eval_host(_policy(policy), P, M, v, cost_f.data_ptr(), cost_b.data_ptr(),
                                None if comm is None else comm.data_ptr(), n, ws.data_ptr(), ws.numel(),
                                host["makespan"].data_ptr(), host["idle"].data_ptr(), host["bub_num"].data_ptr(),
                                host["bub_den"].data_ptr(), host["peak"].data_ptr(), host["status"].data_ptr(),
                                _stream(stream))
    _check(rc, "pp_sched_eval_host")
    h2d = 4 * (2 * S * M * n + (0 if comm is None else max(S - 1, 0) * n))
    d2h = sum(t.numel() * t.element_size() for t in host.values())
    return host, h2d, d2h


def partition_search(layer_tf, layer_tb, layer_act, P, M, comm, cap, seed, cand_begin, n_cand,
                     all_makespan=False, out=None, stream=None):
    """Call pp_sched_partition_search; layer arrays are CUDA tensors (int32,
    int32, int64).  Returns dict(best_idx int64[1], best_makespan int32[1],
    best_cuts int32[P-1], all_makespan int32[n_cand] if requested)."""
    dev = layer_tf.device
    out = dict(out or {})
    bi = out.setdefault("best_idx", torch.empty(1, dtype=torch.int64, device=dev))
    bm = out.setdefault("best_makespan", torch.empty(1, dtype=torch.int32, device=dev))
    bc = out.setdefault("best_cuts", torch.empty(max(P - 1, 1), dtype=torch.int32, device=dev))
    am = None
    if all_makespan:
        am = out.setdefault("all_makespan", torch.empty(n_cand, dtype=torch.int32, device=dev))
    L = layer_tf.numel()
    rc = LIB.pp_sched_partition_search(_ptr(layer_tf), _ptr(layer_tb), _ptr(layer_act), L, P, M,
                                       int(comm), int(cap), ctypes.c_uint64(seed & (2**64 - 1)),
                                       int(cand_begin), int(n_cand), _ptr(bi), _ptr(bm),
                                       _ptr(bc) if P > 1 else None, _ptr(am), _stream(stream))
    _check(rc, "pp_sched_partition_search")
    return out


def partition_search_ranks(layer_tf, layer_tb, layer_act, P, M, comm, cap, rank_begin, n_ranks,
                           all_makespan=False, out=None, stream=None):
    """Call pp_sched_partition_search_ranks (the exhaustive search over colex
    ranks [rank_begin, rank_begin + n_ranks)).  Returns dict(best_idx (the
    winning rank) int64[1], best_makespan, best_cuts, all_makespan if asked)."""
    dev = layer_tf.device
    out = dict(out or {})
    bi = out.setdefault("best_idx", torch.empty(1, dtype=torch.int64, device=dev))
    bm = out.setdefault("best_makespan", torch.empty(1, dtype=torch.int32, device=dev))
    bc = out.setdefault("best_cuts", torch.empty(max(P - 1, 1), dtype=torch.int32, device=dev))
    am = None
    if all_makespan:
        am = out.setdefault("all_makespan", torch.empty(n_ranks, dtype=torch.int32, device=dev))
    L = layer_tf.numel()
    rc = LIB.pp_sched_partition_search_ranks(_ptr(layer_tf), _ptr(layer_tb), _ptr(layer_act), L, P, M,
                                             int(comm), int(cap), int(rank_begin), int(n_ranks), _ptr(bi),
                                             _ptr(bm), _ptr(bc) if P > 1 else None, _ptr(am), _stream(stream))
    _check(rc, "pp_sched_partition_search_ranks")
    return out


def partition_search_interleaved(layer_tf, layer_tb, layer_act, P, v, M, comm, cap, seed, cand_begin, n_cand,
                                 all_makespan=False, out=None, stream=None):
    """Call pp_sched_partition_search_interleaved (S = P*v ranges).  Returns
    dict(best_idx, best_makespan, best_cuts int32[S-1], all_makespan)."""
    dev = layer_tf.device
    out = dict(out or {})
    bi = out.setdefault("best_idx", torch.empty(1, dtype=torch.int64, device=dev))
    bm = out.setdefault("best_makespan", torch.empty(1, dtype=torch.int32, device=dev))
    bc = out.setdefault("best_cuts", torch.empty(P * v - 1, dtype=torch.int32, device=dev))
    am = None
    if all_makespan:
        am = out.setdefault("all_makespan", torch.empty(n_cand, dtype=torch.int32, device=dev))
    L = layer_tf.numel()
    rc = LIB.pp_sched_partition_search_interleaved(_ptr(layer_tf), _ptr(layer_tb), _ptr(layer_act), L, P, v, M,
                                                   int(comm), int(cap), ctypes.c_uint64(seed & (2**64 - 1)),
                                                   int(cand_begin), int(n_cand), _ptr(bi), _ptr(bm), _ptr(bc),
                                                   _ptr(am), _stream(stream))
    _check(rc, "pp_sched_partition_search_interleaved")
    return out


def cache_clear():
    LIB.pp_sched_cache_clear()
