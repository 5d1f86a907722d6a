"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws numbers (NumPy PCG64, fixed seed per workload); it holds
none of the evaluator's arithmetic.  Both the CUDA path and the CPU oracle are
fed from here.  Uniform integer ranges are inclusive.

Cost tables are returned in the GPU's native instance-minor layout,
[virtual stage][microbatch][instance], with element strides
(inst, stage, mb) = (1, M*n, n); an instance-major view is one transpose away.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GPIPE, ONEF1B, INTERLEAVED, ZB1P, ZB2P, GPIPE_FIFO = 0, 1, 2, 3, 4, 5


@dataclass
class Batch:
    """One evaluation call's worth of instances (all of one policy and shape)."""
    policy: int
    P: int
    M: int
    v: int
    n: int
    cost_f: np.ndarray            # int32, flat buffer indexed through `strides`
    cost_b: np.ndarray
    strides: tuple                # element strides (inst, stage, mb)
    comm: np.ndarray | None       # int32, flat buffer indexed through `comm_strides`
    comm_strides: tuple = (0, 0)  # element strides (inst, boundary)
    meta: dict = field(default_factory=dict)
    cost_w: np.ndarray | None = None  # Zero Bubble only: W costs, same strides as cost_f

    @property
    def S(self):
        return self.P * self.v

    @property
    def op_times(self):
        return (3 if self.cost_w is not None else 2) * self.P * self.M * self.v * self.n


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def uniform_batch(policy, P, M, v, tf, tb, comm):
    """Instances whose costs are one scalar t_f / t_b per instance (strides 0 over
    stage and microbatch) and one comm value per instance on every boundary."""
    tf = np.ascontiguousarray(tf, np.int32).reshape(-1)
    tb = np.ascontiguousarray(tb, np.int32).reshape(-1)
    n = tf.shape[0]
    cm = None if comm is None else np.ascontiguousarray(comm, np.int32).reshape(-1)
    return Batch(policy, P, M, v, n, tf, tb, (1, 0, 0), cm, (1, 0))


def worked_examples():
    """Single instances: P=4, M=8, t_f=1, t_b=2, comm 0 (GPipe and 1F1B), and the
    two-stage, four-microbatch worked case with t_f = t_b = 1."""
    out = []
    for policy in (GPIPE, ONEF1B):
        out.append(uniform_batch(policy, 4, 8, 1, [1], [2], [0]))
        out.append(uniform_batch(policy, 2, 4, 1, [1], [1], [0]))
    return out


def sweep_shapes():
    """The closed-form sweep's shapes: P in 2..16 x M in 1..128 for GPipe and 1F1B,
    interleaved v=2 where P divides M."""
    shapes = []
    for P in range(2, 17):
        for M in range(1, 129):
            shapes.append((GPIPE, P, M, 1))
            shapes.append((ONEF1B, P, M, 1))
            if M % P == 0:
                shapes.append((INTERLEAVED, P, M, 2))
    return shapes


def sweep_batch(policy, P, M, v):
    """All 16 combinations of t_f in {1..4}, t_b in {t_f, 2 t_f}, comm in {0, 1}
    for one shape, one instance each."""
    tf, tb, cm = [], [], []
    for f in (1, 2, 3, 4):
        for b in (f, 2 * f):
            for c in (0, 1):
                tf.append(f); tb.append(b); cm.append(c)
    return uniform_batch(policy, P, M, v, tf, tb, cm)


def hetero_1f1b(n=65536, seed=3, P=8, M=64):
    """Heterogeneous 1F1B batch: per (instance, stage, microbatch) t_f ~ U[80,120],
    t_b ~ U[160,240]; comm ~ U[2,8] per (instance, boundary)."""
    rng = _rng(seed)
    cf = rng.integers(80, 120, size=(P, M, n), dtype=np.int32, endpoint=True)
    cb = rng.integers(160, 240, size=(P, M, n), dtype=np.int32, endpoint=True)
    cm = rng.integers(2, 8, size=(max(P - 1, 1), n), dtype=np.int32, endpoint=True)
    return Batch(ONEF1B, P, M, 1, n, cf.reshape(-1), cb.reshape(-1), (1, M * n, n),
                 cm.reshape(-1), (1, n), meta={"workload": f"1f1b_hetero_P{P}_M{M}_n{n}"})


def interleaved_vs_1f1b(v, n=16384, seed=4, P=8, M=128):
    """Interleaved batch: per (instance, virtual stage) t_f ~ U[40,60],
    t_b = 2 t_f + U[-5,5], comm = 3, costs broadcast over microbatches
    (stride_mb = 0).  Also returns the 1F1B batch with the same total work per
    device: stage k's cost is the sum over the device's chunks."""
    rng = _rng(seed * 100 + v)
    S = P * v
    tf = rng.integers(40, 60, size=(S, n), dtype=np.int32, endpoint=True)
    tb = (2 * tf + rng.integers(-5, 5, size=(S, n), dtype=np.int32, endpoint=True)).astype(np.int32)
    cm = np.full((S - 1, n), 3, np.int32)
    il = Batch(INTERLEAVED, P, M, v, n, tf.reshape(-1), tb.reshape(-1), (1, n, 0),
               cm.reshape(-1), (1, n), meta={"workload": f"interleaved_P{P}_v{v}_M{M}_n{n}"})
    tf1 = tf.reshape(v, P, n).sum(axis=0).astype(np.int32)
    tb1 = tb.reshape(v, P, n).sum(axis=0).astype(np.int32)
    cm1 = np.full((P - 1, n), 3, np.int32)
    base = Batch(ONEF1B, P, M, 1, n, tf1.reshape(-1), tb1.reshape(-1), (1, n, 0),
                 cm1.reshape(-1), (1, n), meta={"workload": f"1f1b_equal_work_P{P}_M{M}_n{n}"})
    return il, base


@dataclass
class SearchProblem:
    layer_tf: np.ndarray   # int32 [L]
    layer_tb: np.ndarray   # int32 [L]
    layer_act: np.ndarray  # int64 [L], bytes
    P: int
    M: int
    comm: int
    cap: int
    seed: int
    n_cand: int


def layer_split(seed=5, L=80, P=8, M=128, n_cand=1 << 20):
    """80-layer model: per-layer t_f = u ~ U[90,110] ticks, the embedding layer
    (layer 0) floor(1.5 u), the output projection (layer L-1) 3u, t_b = 2 t_f;
    activation bytes ~ U[200,300] * 10^6; cap 80 * 10^9 bytes; comm 0."""
    rng = _rng(seed)
    u = rng.integers(90, 110, size=L, dtype=np.int64, endpoint=True)
    tf = u.copy()
    tf[0] = (3 * u[0]) // 2
    tf[L - 1] = 3 * u[L - 1]
    act = rng.integers(200, 300, size=L, dtype=np.int64, endpoint=True) * 10**6
    return SearchProblem(tf.astype(np.int32), (2 * tf).astype(np.int32), act, P, M, 0,
                         80 * 10**9, int(rng.integers(0, 2**63 - 1)), n_cand)


def random_batch(policy, P, M, v, n, seed, lo=0, hi=9, comm_hi=4, layout="inst_minor",
                 stride_mb_zero=False, pad_to=1):
    """Small random instances for parity tests (any policy/shape/layout).

    With the instance-minor layout each (stage, microbatch) row holds n
    instances padded to a multiple of `pad_to` elements (the pad is zero)."""
    rng = _rng(seed)
    S = P * v
    Mx = 1 if stride_mb_zero else M
    cf = rng.integers(lo, hi, size=(n, S, Mx), dtype=np.int32, endpoint=True)
    cb = rng.integers(lo, hi, size=(n, S, Mx), dtype=np.int32, endpoint=True)
    cm = rng.integers(0, comm_hi, size=(n, max(S - 1, 1)), dtype=np.int32, endpoint=True)
    if layout == "inst_minor":
        pitch = -(-n // pad_to) * pad_to if n else 0
        rows_f = np.zeros((S, Mx, pitch), np.int32)
        rows_b = np.zeros((S, Mx, pitch), np.int32)
        rows_f[:, :, :n] = np.transpose(cf, (1, 2, 0))
        rows_b[:, :, :n] = np.transpose(cb, (1, 2, 0))
        cfa, cba = rows_f.reshape(-1), rows_b.reshape(-1)
        st = (1, Mx * pitch, 0 if stride_mb_zero else pitch)
        cma = np.ascontiguousarray(cm.T).reshape(-1)
        cst = (1, n)
    else:
        cfa, cba = cf.reshape(-1), cb.reshape(-1)
        st = (S * Mx, Mx, 0 if stride_mb_zero else 1)
        cma = cm.reshape(-1)
        cst = (max(S - 1, 1), 1)
    return Batch(policy, P, M, v, n, cfa, cba, st, cma, cst)


def hetero_zb(policy=ZB1P, n=65536, seed=6, P=8, M=64):
    """Heterogeneous Zero Bubble batch: the 1F1B batch's t_b ~ U[160,240] split
    into B ~ U[80,120] and W ~ U[80,120]; t_f ~ U[80,120]; comm ~ U[2,8];
    instance-minor layout."""
    rng = _rng(seed)
    cf = rng.integers(80, 120, size=(P, M, n), dtype=np.int32, endpoint=True)
    cb = rng.integers(80, 120, size=(P, M, n), dtype=np.int32, endpoint=True)
    cw = rng.integers(80, 120, size=(P, M, n), dtype=np.int32, endpoint=True)
    cm = rng.integers(2, 8, size=(max(P - 1, 1), n), dtype=np.int32, endpoint=True)
    name = "zb1p" if policy == ZB1P else "zb2p"
    return Batch(policy, P, M, 1, n, cf.reshape(-1), cb.reshape(-1), (1, M * n, n), cm.reshape(-1), (1, n),
                 meta={"workload": f"{name}_hetero_P{P}_M{M}_n{n}"}, cost_w=cw.reshape(-1))


def hetero_dualpipe(n=65536, seed=7, P=8, M=64):
    """Heterogeneous DualPipe batch: the 1F1B batch's distributions (t_f ~
    U[80,120], t_b ~ U[160,240] per (instance, block, microbatch), comm ~
    U[2,8] per (instance, link)), half of the microbatches on each route."""
    b = hetero_1f1b(n=n, seed=seed, P=P, M=M)
    b.meta = {"workload": f"dualpipe_hetero_P{P}_M{M}_n{n}", "m_a": (M + 1) // 2}
    return b


def random_zb(policy, P, M, n, seed, lo=1, hi=9, w_lo=0, w_hi=9, comm_hi=4, layout="inst_minor", pad_to=1):
    """Small random Zero Bubble instances for parity tests (F, B in [lo, hi],
    W in [w_lo, w_hi], comm in [0, comm_hi])."""
    rng = _rng(seed)
    cf = rng.integers(lo, hi, size=(n, P, M), dtype=np.int32, endpoint=True)
    cb = rng.integers(lo, hi, size=(n, P, M), dtype=np.int32, endpoint=True)
    cw = rng.integers(w_lo, w_hi, size=(n, P, M), dtype=np.int32, endpoint=True)
    cm = rng.integers(0, comm_hi, size=(n, max(P - 1, 1)), dtype=np.int32, endpoint=True)
    if layout == "inst_minor":
        pitch = -(-n // pad_to) * pad_to if n else 0
        arrs = []
        for c in (cf, cb, cw):
            rows = np.zeros((P, M, pitch), np.int32)
            rows[:, :, :n] = np.transpose(c, (1, 2, 0))
            arrs.append(rows.reshape(-1))
        st = (1, M * pitch, pitch)
        cma = np.ascontiguousarray(cm.T).reshape(-1)
        cst = (1, n)
    else:
        arrs = [c.reshape(-1) for c in (cf, cb, cw)]
        st = (P * M, M, 1)
        cma = cm.reshape(-1)
        cst = (max(P - 1, 1), 1)
    return Batch(policy, P, M, 1, n, arrs[0], arrs[1], st, cma, cst, cost_w=arrs[2])
