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
           "pp_sched_many_info", "pp_sched_many_destroy", "pp_sched_eval_dualpipe", "pp_sched_debug_checks")


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
    # PPSCHED_CHECKED=1 loads the bounds-checked build (build_lib.build(checked=True))
    checked = os.environ.get("PPSCHED_CHECKED", "0") not in ("", "0")
    path = build_lib.LIB_CHECKED if checked else build_lib.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"{os.path.basename(path)} is not built ({path}); run __graft_entry__.build() or "
            "python -m pipeline_schedule_simulation_gb300.build_lib" + (" --checked" if checked else ""))
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
    lib.pp_sched_debug_checks.argtypes = [vp]
    lib.pp_sched_debug_checks.restype = i32
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


def _reach(count, strides):
    """Elements a strided access reaches from its base pointer: 1 + the largest
    offset sum((extent - 1) * stride), or 0 when any extent is 0.  `count` and
    `strides` pair each extent with its element stride."""
    r = 1
    for c, st in zip(count, strides):
        if c <= 0:
            return 0
        r += (c - 1) * st
    return r


def _avail(t):
    """Elements of t's storage from its data pointer on."""
    return t.untyped_storage().nbytes() // t.element_size() - t.storage_offset()


def _arg(t, name, dtype, device, reach, host=False):
    """Refuse, before any library call, a buffer the library would address
    wrongly: not a tensor, on the wrong device (CUDA device `device`, or the
    CPU for host inputs), of the wrong dtype, or too short for the `reach`
    elements its strides address from its data pointer (the library reads raw
    pointers and element strides, not the tensor's own shape)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if host:
        if t.is_cuda:
            raise ValueError(f"{name}: expected a host (CPU) tensor, got one on {t.device}")
    elif not t.is_cuda or (device is not None and t.device != device):
        raise ValueError(f"{name}: expected a tensor on {device or 'a CUDA device'}, got one on {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected dtype {dtype}, got {t.dtype}")
    # a contiguous tensor of at least `reach` elements holds them from its data
    # pointer; otherwise ask its storage
    if reach > 0 and not (t.numel() >= reach and t.is_contiguous()):
        avail = _avail(t)
        if reach > avail:
            raise ValueError(f"{name}: the strides reach {reach} elements from its data pointer but its storage "
                             f"holds {avail}")
    return t


def _inputs(P, M, v, S, cost_tensors, strides, n, comm_tensors, comm_strides):
    """Check the cost tables (int32, indexed (instance, stage, microbatch)) and
    the comm tables (int32, (instance, boundary)) of one evaluation; returns
    their device."""
    dev = next((t.device for _, t in cost_tensors if isinstance(t, torch.Tensor) and t.is_cuda), None)
    if len(strides) != 3 or len(comm_strides) != 2:
        raise ValueError("strides must be (inst, stage, mb) and comm_strides (inst, boundary)")
    if min(int(x) for x in strides) < 0 or min(int(x) for x in comm_strides) < 0:
        raise ValueError("strides must be non-negative")
    reach = _reach((n, S, M), strides)
    for name, t in cost_tensors:
        if t is not None:  # a missing table is the library's argument error
            _arg(t, name, torch.int32, dev, reach)
    creach = _reach((n, S - 1), comm_strides)
    for name, t in comm_tensors:
        if t is not None:
            _arg(t, name, torch.int32, dev, creach)
    return dev


def _check_outputs(out, n, P, op_count, op_strides, op_names, peak_per_instance=False):
    """The summary outputs hold n (makespan, bub_num, bub_den, status), n*P
    (idle) and P or n*P (peak) elements; the per-op outputs reach what their
    (instance, op) strides address."""
    if n > 0:
        for k, need in (("makespan", n), ("bub_num", n), ("bub_den", n), ("status", n), ("idle", n * P),
                        ("peak", n * P if peak_per_instance else P)):
            t = out.get(k)
            if t is not None and not (t.numel() >= need and t.is_contiguous()) and need > _avail(t):
                raise ValueError(f"{k}: needs {need} elements, its storage holds {_avail(t)}")
    for k in op_names:
        t = out.get(k)
        if t is not None:
            reach = _reach(op_count, op_strides)
            if not (t.numel() >= reach and t.is_contiguous()) and reach > _avail(t):
                raise ValueError(f"{k}: the op strides reach {reach} elements, its storage holds {_avail(t)}")


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
    dev = _inputs(P, M, v, P * v, (("cost_f", cost_f), ("cost_b", cost_b)), strides, n,
                  (("comm", comm), ("comm_b", comm_b)), comm_strides)
    out = dict(out or {})
    O = 2 * M * v

    def want(name, shape, dtype):
        if name in out:
            return _arg(out[name], name, dtype, dev, 0)
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
        _check_outputs(out, n, P, (n, P * O), op_strides, ("op_start", "op_end"))
    else:
        op_strides = (0, 0)
    _check_outputs(out, n, P, None, None, ())
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
    dev = _inputs(P, M, 1, P, (("cost_f", cost_f), ("cost_b", cost_b)), strides, n, (("comm", comm),),
                  comm_strides)
    out = dict(out or {})

    def want(name, shape, dtype):
        if name in out:
            return _arg(out[name], name, dtype, dev, 0)
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
        _check_outputs(out, n, P, (n, P * 2 * M), op_strides, ("op_start", "op_end"), True)
    else:
        op_strides = (0, 0)
    _check_outputs(out, n, P, None, None, (), True)
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
    dev = _inputs(P, M, 1, P, (("cost_f", cost_f), ("cost_b", cost_b), ("cost_w", cost_w)), strides, n,
                  (("comm", comm),), comm_strides)
    out = dict(out or {})

    def want(name, shape, dtype):
        if name in out:
            return _arg(out[name], name, dtype, dev, 0)
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
        _check_outputs(out, n, P, (n, P * 3 * M), op_strides, ("op_start", "op_end"), True)
    else:
        op_strides = (0, 0)
    _check_outputs(out, n, P, None, None, (), True)
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
            comm = q.get("comm")
            cs = q.get("comm_strides", (0, 0))
            v = q.get("v", 1)
            dev = _inputs(P, q["M"], v, P * v, (("cost_f", q["cost_f"]), ("cost_b", q["cost_b"])), q["strides"],
                          n, (("comm", comm),), cs)
            for k, shape, dt in (("makespan", (n,), torch.int32), ("idle", (n, P), torch.int32),
                                 ("bub_num", (n,), torch.int64), ("bub_den", (n,), torch.int64),
                                 ("peak", (P,), torch.int32), ("status", (n,), torch.int8)):
                if k not in out:
                    out[k] = torch.empty(shape, dtype=dt, device=dev)
                else:
                    _arg(out[k], k, dt, dev, 0)
            _check_outputs(out, n, P, None, None, ())
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
    for name, t, count in (("cost_f", cost_f, S * M * n), ("cost_b", cost_b, S * M * n),
                           ("comm", comm, max(S - 1, 0) * n)):
        if t is not None:
            _arg(t, name, torch.int32, None, count, host=True)
            if not t.is_contiguous():
                raise ValueError(f"{name}: the host entry reads a contiguous [S][M][n] table")
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


def _layers(layer_tf, layer_tb, layer_act):
    """The per-layer tables of a search: int32 t_f and t_b, int64 activation
    bytes, one entry per layer, on one CUDA device; returns (L, device)."""
    L = layer_tf.numel() if isinstance(layer_tf, torch.Tensor) else 0
    dev = layer_tf.device if isinstance(layer_tf, torch.Tensor) and layer_tf.is_cuda else None
    _arg(layer_tf, "layer_tf", torch.int32, dev, L)
    _arg(layer_tb, "layer_tb", torch.int32, dev, L)
    _arg(layer_act, "layer_act", torch.int64, dev, L)
    return L, dev


def _search_outputs(bi, bm, bc, am, ncuts, ncand, dev):
    _arg(bi, "best_idx", torch.int64, dev, 1)
    _arg(bm, "best_makespan", torch.int32, dev, 1)
    _arg(bc, "best_cuts", torch.int32, dev, ncuts)
    if am is not None:
        _arg(am, "all_makespan", torch.int32, dev, ncand)


def partition_search(layer_tf, layer_tb, layer_act, P, M, comm, cap, seed, cand_begin, n_cand,
                     all_makespan=False, out=None, stream=None):
    """Call pp_sched_partition_search; layer arrays are CUDA tensors (int32,
    int32, int64).  Returns dict(best_idx int64[1], best_makespan int32[1],
    best_cuts int32[P-1], all_makespan int32[n_cand] if requested)."""
    L, dev = _layers(layer_tf, layer_tb, layer_act)
    out = dict(out or {})
    bi = out.setdefault("best_idx", torch.empty(1, dtype=torch.int64, device=dev))
    bm = out.setdefault("best_makespan", torch.empty(1, dtype=torch.int32, device=dev))
    bc = out.setdefault("best_cuts", torch.empty(max(P - 1, 1), dtype=torch.int32, device=dev))
    am = None
    if all_makespan:
        am = out.setdefault("all_makespan", torch.empty(n_cand, dtype=torch.int32, device=dev))
    _search_outputs(bi, bm, bc, am, max(P - 1, 1), n_cand, dev)
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
    L, dev = _layers(layer_tf, layer_tb, layer_act)
    out = dict(out or {})
    bi = out.setdefault("best_idx", torch.empty(1, dtype=torch.int64, device=dev))
    bm = out.setdefault("best_makespan", torch.empty(1, dtype=torch.int32, device=dev))
    bc = out.setdefault("best_cuts", torch.empty(max(P - 1, 1), dtype=torch.int32, device=dev))
    am = None
    if all_makespan:
        am = out.setdefault("all_makespan", torch.empty(n_ranks, dtype=torch.int32, device=dev))
    _search_outputs(bi, bm, bc, am, max(P - 1, 1), n_ranks, dev)
    rc = LIB.pp_sched_partition_search_ranks(_ptr(layer_tf), _ptr(layer_tb), _ptr(layer_act), L, P, M,
                                             int(comm), int(cap), int(rank_begin), int(n_ranks), _ptr(bi),
                                             _ptr(bm), _ptr(bc) if P > 1 else None, _ptr(am), _stream(stream))
    _check(rc, "pp_sched_partition_search_ranks")
    return out


def partition_search_interleaved(layer_tf, layer_tb, layer_act, P, v, M, comm, cap, seed, cand_begin, n_cand,
                                 all_makespan=False, out=None, stream=None):
    """Call pp_sched_partition_search_interleaved (S = P*v ranges).  Returns
    dict(best_idx, best_makespan, best_cuts int32[S-1], all_makespan)."""
    L, dev = _layers(layer_tf, layer_tb, layer_act)
    out = dict(out or {})
    bi = out.setdefault("best_idx", torch.empty(1, dtype=torch.int64, device=dev))
    bm = out.setdefault("best_makespan", torch.empty(1, dtype=torch.int32, device=dev))
    bc = out.setdefault("best_cuts", torch.empty(P * v - 1, dtype=torch.int32, device=dev))
    am = None
    if all_makespan:
        am = out.setdefault("all_makespan", torch.empty(n_cand, dtype=torch.int32, device=dev))
    _search_outputs(bi, bm, bc, am, P * v - 1, n_cand, dev)
    rc = LIB.pp_sched_partition_search_interleaved(_ptr(layer_tf), _ptr(layer_tb), _ptr(layer_act), L, P, v, M,
                                                   int(comm), int(cap), ctypes.c_uint64(seed & (2**64 - 1)),
                                                   int(cand_begin), int(n_cand), _ptr(bi), _ptr(bm), _ptr(bc),
                                                   _ptr(am), _stream(stream))
    _check(rc, "pp_sched_partition_search_interleaved")
    return out


def cache_clear():
    LIB.pp_sched_cache_clear()


def debug_checks():
    """(checked build?, first failure word since the last call or 0); see
    pp_sched_debug_checks.  Synchronizes the device."""
    w = ctypes.c_uint64(0)
    checked = LIB.pp_sched_debug_checks(ctypes.byref(w))
    return bool(checked), int(w.value)
