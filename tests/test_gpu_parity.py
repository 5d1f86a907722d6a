"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle,
element by element, bit-exact (all quantities are integers; the bubble's float
view is checked to 1e-12)."""
import os

import numpy as np
import pytest

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import assert_same, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

NCPU = os.cpu_count() or 8


@pytest.fixture(scope="module")
def B():
    from pipeline_schedule_simulation_gb300 import binding
    return binding


def test_worked_examples_every_op(orc, B):
    for batch in W.worked_examples():
        g = run_gpu(batch, op_times=True)
        r = run_oracle(orc, batch, op_times=True)
        assert_same(g, r, op_times=True)
    # the worked 2x4 tables end in 10 units; P=4 M=8 t_f=1 t_b=2 in 33 with bubble 36/132
    g = run_gpu(W.uniform_batch(W.ONEF1B, 4, 8, 1, [1], [2], [0]))
    assert g["makespan"][0] == 33 and g["bub_num"][0] == 36 and g["bub_den"][0] == 132
    assert list(g["peak"]) == [4, 3, 2, 1]


def test_plan_tables_match_oracle(orc, B):
    for policy, P, M, v in [(0, 4, 8, 1), (1, 4, 8, 1), (1, 8, 3, 1), (2, 4, 8, 2), (2, 8, 16, 4),
                            (1, 16, 128, 1), (2, 3, 6, 3), (1, 1, 5, 1), (2, 1, 3, 4)]:
        plan = B.Plan(policy, P, M, v)
        ops, peak, rnd = plan.tables()
        kind, chunk, mb = B.op_fields(ops)
        okind, ochunk, omb = orc.order(policy, P, M, v)
        assert np.array_equal(kind.numpy(), okind)
        assert np.array_equal(chunk.numpy(), ochunk)
        assert np.array_equal(mb.numpy(), omb)
        # rounds are the start ticks at unit cost and zero comm
        ref = orc.evaluate(policy, P, M, v, 1, 1)
        assert np.array_equal(rnd.numpy(), ref["start"])
        assert np.array_equal(peak.numpy(), ref["peak"])
        assert plan.rounds == ref["makespan"]
        assert plan.register_path == (1 if v == 1 else 0)


SHAPES = [
    (W.GPIPE, 1, 1, 1), (W.ONEF1B, 1, 7, 1), (W.GPIPE, 2, 4, 1), (W.ONEF1B, 3, 2, 1),
    (W.ONEF1B, 4, 8, 1), (W.GPIPE, 5, 13, 1), (W.ONEF1B, 8, 3, 1), (W.ONEF1B, 8, 64, 1),
    (W.GPIPE, 8, 64, 1), (W.ONEF1B, 12, 20, 1), (W.ONEF1B, 16, 40, 1), (W.GPIPE, 16, 9, 1),
    (W.INTERLEAVED, 2, 4, 2), (W.INTERLEAVED, 4, 8, 2), (W.INTERLEAVED, 3, 9, 3),
    (W.INTERLEAVED, 8, 16, 4), (W.INTERLEAVED, 16, 32, 2), (W.INTERLEAVED, 1, 3, 5),
    (W.GPIPE_FIFO, 1, 4, 1), (W.GPIPE_FIFO, 3, 7, 1), (W.GPIPE_FIFO, 8, 16, 1), (W.GPIPE_FIFO, 16, 5, 1),
]


@pytest.mark.parametrize("policy,P,M,v", SHAPES)
@pytest.mark.parametrize("layout", ["inst_minor", "inst_major"])
def test_random_batches(orc, B, policy, P, M, v, layout):
    # several warps and a ragged tail: n = 32*k + r
    for n, seed, mbz in ((77, 1, False), (161, 2, True)):
        batch = W.random_batch(policy, P, M, v, n, seed=seed + 10 * P + M, hi=12, comm_hi=5,
                               layout=layout, stride_mb_zero=mbz)
        g = run_gpu(batch, op_times=True)
        r = run_oracle(orc, batch, op_times=True)
        assert_same(g, r, op_times=True)


VEC_SHAPES = [
    (W.INTERLEAVED, 8, 16, 2), (W.INTERLEAVED, 4, 8, 3), (W.INTERLEAVED, 16, 32, 2),
    (W.INTERLEAVED, 2, 4, 4), (W.INTERLEAVED, 3, 6, 2), (W.ONEF1B, 8, 12, 1), (W.GPIPE, 4, 8, 1),
]


@pytest.mark.parametrize("policy,P,M,v", VEC_SHAPES)
def test_vector_rows_ragged_tail(orc, B, policy, P, M, v):
    """Instance-minor rows padded to 16 bytes take the vector loaders; n
    leaves a last copy that covers fewer instances than its width."""
    for n, seed in ((77, 5), (161, 6), (3, 7)):
        batch = W.random_batch(policy, P, M, v, n, seed=seed + P + M, hi=12, comm_hi=5, pad_to=4)
        assert batch.strides[1] % 4 == 0 and batch.strides[2] % 4 == 0
        g = run_gpu(batch, op_times=True)
        r = run_oracle(orc, batch, op_times=True)
        assert_same(g, r, op_times=True)


@pytest.mark.parametrize("P,M,v,n", [(4, 4, 2, 19456 + 37), (8, 8, 2, 9728 + 13), (16, 16, 2, 4864 + 3),
                                     (3, 6, 3, 19456 + 5)])
@pytest.mark.parametrize("layout", ["inst_minor", "inst_major"])
def test_interleaved_two_sets_per_lane(orc, B, P, M, v, n, layout):
    """Batches large enough for the lane evaluator's two-instance-set layout
    (about eight warps per SM), with a ragged last warp, every op time."""
    batch = W.random_batch(W.INTERLEAVED, P, M, v, n, seed=P * 100 + M, hi=30, comm_hi=6, layout=layout, pad_to=4)
    g = run_gpu(batch, op_times=True)
    r = run_oracle(orc, batch, op_times=True)
    assert_same(g, r, op_times=True)


def test_status_interleaved(orc, B):
    P, M, v, n = 4, 8, 2, 70
    S = P * v
    batch = W.random_batch(W.INTERLEAVED, P, M, v, n, seed=9, layout="inst_major")
    cf = batch.cost_f.reshape(n, S, M)
    cb = batch.cost_b.reshape(n, S, M)
    cf[3, 5, 2] = -1
    cb[10, 0, 0] = 2**31 - 1
    cf[11, 7, 7] = 2**30
    cb[11, 2, 3] = 2**30
    batch.comm.reshape(n, S - 1)[20, 4] = -4
    batch.comm.reshape(n, S - 1)[21, 6] = 2**31 - 2
    g = run_gpu(batch)
    r = run_oracle(orc, batch)
    assert g["status"][3] == B.ST_NEG_COST and g["status"][20] == B.ST_NEG_COST
    assert g["status"][10] == B.ST_OVERFLOW and g["status"][21] == B.ST_OVERFLOW
    assert_same(g, r)


def test_generic_evaluator_wide_strides(orc, B):
    """Cost rows more than 2^30 elements apart are beyond the lane
    evaluator's loader table, so interleaved instances run on the generic
    slot evaluator: same numbers.  Forward and backward costs share one
    sparse 8 GB buffer (backward rows sit n*M elements after forward rows)."""
    import torch
    P, M, v, n = 8, 8, 4, 40
    S = P * v
    compact = W.random_batch(W.INTERLEAVED, P, M, v, n, seed=12, hi=12, comm_hi=5, layout="inst_major")
    si, ss, sm = M, 1 << 26, 1
    assert (S - 1) * ss >= 1 << 30
    x, s, m = np.meshgrid(np.arange(n), np.arange(S), np.arange(M), indexing="ij")
    idx = (x * si + s * ss + m * sm).reshape(-1)
    buf = torch.empty(int(idx.max()) + n * M + 1, dtype=torch.int32, device="cuda")
    buf[torch.from_numpy(idx).cuda()] = to_dev(compact.cost_f.reshape(-1))
    buf[torch.from_numpy(idx + n * M).cuda()] = to_dev(compact.cost_b.reshape(-1))
    out = B.evaluate(W.INTERLEAVED, P, M, v, buf, buf[n * M:], (si, ss, sm), n, comm=to_dev(compact.comm),
                     comm_strides=compact.comm_strides, op_times=True)
    torch.cuda.synchronize()
    g = {k: t.cpu().numpy() for k, t in out.items()}
    del buf, out
    torch.cuda.empty_cache()
    r = run_oracle(orc, compact, op_times=True)
    assert_same(g, r, op_times=True)


def test_zero_costs_and_empty(orc, B):
    batch = W.random_batch(W.ONEF1B, 4, 6, 1, 40, seed=3, lo=0, hi=0, comm_hi=0)
    g = run_gpu(batch)
    assert (g["makespan"] == 0).all() and (g["bub_den"] == 0).all() and (g["bub_num"] == 0).all()
    r = run_oracle(orc, batch)
    assert_same(g, r)
    empty = W.random_batch(W.ONEF1B, 4, 6, 1, 0, seed=3)
    out = B.evaluate(1, 4, 6, 1, to_dev(np.zeros(4, np.int32)), to_dev(np.zeros(4, np.int32)),
                     empty.strides, 0)
    assert out["makespan"].numel() == 0


def test_status_negative_and_overflow(orc, B):
    batch = W.random_batch(W.ONEF1B, 4, 8, 1, 70, seed=4, layout="inst_major")
    cf = batch.cost_f.reshape(70, 4, 8)
    cb = batch.cost_b.reshape(70, 4, 8)
    cf[3, 2, 5] = -1
    cb[10, 0, 0] = 2**31 - 1
    cb[11, 3, 7] = 2**30
    cf[11, 0, 0] = 2**30
    batch.comm.reshape(70, 3)[20, 1] = -4
    batch.comm.reshape(70, 3)[21, 1] = 2**31 - 2
    g = run_gpu(batch)
    r = run_oracle(orc, batch)
    assert g["status"][3] == B.ST_NEG_COST and g["status"][20] == B.ST_NEG_COST
    assert g["status"][10] == B.ST_OVERFLOW and g["status"][21] == B.ST_OVERFLOW
    assert_same(g, r)


def test_closed_form_sweep(orc, B):
    """Every shape of the closed-form sweep (GPipe, 1F1B, interleaved v=2),
    every instance: bit-exact against the oracle and equal to the pages'
    closed forms where they exist."""
    from fractions import Fraction
    for policy, P, M, v in W.sweep_shapes():
        batch = W.sweep_batch(policy, P, M, v)
        g = run_gpu(batch)
        tf = batch.cost_f
        tb = batch.cost_b
        cm = batch.comm
        if policy != W.INTERLEAVED:
            base = (M + P - 1) * (tf.astype(np.int64) + tb)
            nocomm = cm == 0
            assert np.array_equal(g["makespan"][nocomm], base[nocomm])
            if policy == W.GPIPE:
                assert np.array_equal(g["makespan"], base + 2 * (P - 1) * cm)
        else:
            sel = (cm == 0) & (tf == tb)
            for x in np.nonzero(sel)[0]:
                assert Fraction(int(g["bub_num"][x]), int(g["bub_den"][x])) == Fraction(P - 1, v * M + P - 1)
        r = run_oracle(orc, batch, nthreads=NCPU)
        assert_same(g, r)


def test_hetero_1f1b_full_batch(orc, B):
    """65,536 heterogeneous 1F1B instances (P=8, M=64) in the benchmark's
    launch configuration: every instance against the oracle, plus invariants."""
    batch = W.hetero_1f1b()
    g = run_gpu(batch)
    r = run_oracle(orc, batch, nthreads=NCPU)
    assert_same(g, r)
    assert (g["status"] == 0).all()
    # invariants for all: busy = makespan - idle equals the summed costs
    cf = batch.cost_f.reshape(8, 64, batch.n).astype(np.int64)
    cb = batch.cost_b.reshape(8, 64, batch.n).astype(np.int64)
    busy = (cf.sum(axis=1) + cb.sum(axis=1)).T
    assert np.array_equal(g["makespan"][:, None] - g["idle"], busy)
    assert np.array_equal(g["bub_num"], g["idle"].astype(np.int64).sum(axis=1))
    assert np.array_equal(g["bub_den"], 8 * g["makespan"].astype(np.int64))
    # a lower bound every valid schedule meets: stage 0's own work plus the
    # first microbatch's round trip
    assert (g["makespan"] >= busy[:, 0]).all()


@pytest.mark.parametrize("v", [2, 4])
def test_interleaved_batches_full(orc, B, v):
    """16,384 interleaved instances (P=8, M=128) and the 1F1B batch with the
    same work per device: every instance against the oracle."""
    il, base = W.interleaved_vs_1f1b(v)
    for batch in (il, base):
        g = run_gpu(batch)
        r = run_oracle(orc, batch, nthreads=NCPU)
        assert_same(g, r)
        assert (g["status"] == 0).all()


def test_split_call_equals_whole(orc, B):
    """Sharding by instance range (one GPU, two calls) gives the same numbers."""
    batch = W.hetero_1f1b(n=4096)
    whole = run_gpu(batch)
    import torch
    cf, cb, cm = to_dev(batch.cost_f), to_dev(batch.cost_b), to_dev(batch.comm)
    half = batch.n // 2
    parts = []
    for lo, hi in ((0, half), (half, batch.n)):
        out = B.evaluate(batch.policy, 8, 64, 1, cf[lo:], cb[lo:], batch.strides, hi - lo,
                         comm=cm[lo:], comm_strides=batch.comm_strides)
        parts.append({k: t.cpu().numpy() for k, t in out.items()})
    torch.cuda.synchronize()
    for k in ("makespan", "idle", "bub_num", "bub_den", "status"):
        assert np.array_equal(np.concatenate([p[k] for p in parts]), whole[k])


@pytest.mark.parametrize("policy,P,M,v,n,ws", [(W.ONEF1B, 8, 64, 1, 1000, None), (W.ONEF1B, 8, 64, 1, 1000, 200_000),
                                               (W.INTERLEAVED, 4, 8, 2, 333, 40_000), (W.GPIPE, 3, 5, 1, 77, None),
                                               (W.ONEF1B, 4, 6, 1, 30, None), (W.ONEF1B, 8, 64, 1, 20000, None)])
def test_host_entry_end_to_end(orc, B, policy, P, M, v, n, ws):
    """pp_sched_eval_host from pinned host buffers, two calls in a row: one
    chunk (n <= 32), chunks one after another (a workspace with room for one
    32-instance slot), or the two-slot pipeline over two streams (the default
    workspace, and a small one with room for two slots), against the oracle."""
    import torch
    if policy == W.ONEF1B and P == 8:
        batches = [W.hetero_1f1b(n=n, seed=s) for s in (3, 4)]
    else:
        batches = [W.random_batch(policy, P, M, v, n, seed=n + s, hi=20, comm_hi=5) for s in (0, 1)]
    staging = {}
    for batch in batches:
        host, h2d, d2h = B.evaluate_host(batch.policy, P, M, v, torch.from_numpy(batch.cost_f).pin_memory(),
                                         torch.from_numpy(batch.cost_b).pin_memory(), batch.n,
                                         comm=torch.from_numpy(batch.comm).pin_memory(), staging=staging,
                                         workspace_bytes=ws)
        torch.cuda.synchronize()
        assert h2d == batch.cost_f.nbytes * 2 + batch.comm.nbytes
        r = run_oracle(orc, batch)
        g = {k: t.numpy().copy() for k, t in host.items()}
        assert_same(g, r)
    if ws is not None:
        assert ws < B.LIB.pp_sched_eval_host_workspace(P, M, v, n)   # really several chunks


FB_SHAPES = [(W.GPIPE, 4, 8, 1), (W.ONEF1B, 8, 16, 1), (W.ONEF1B, 3, 2, 1), (W.GPIPE_FIFO, 5, 6, 1),
             (W.INTERLEAVED, 4, 8, 2), (W.INTERLEAVED, 8, 16, 3), (W.ONEF1B, 16, 20, 1)]


@pytest.mark.parametrize("policy,P,M,v", FB_SHAPES)
@pytest.mark.parametrize("layout", ["inst_minor", "inst_major"])
def test_separate_backward_comm(orc, B, policy, P, M, v, layout):
    """pp_sched_eval_fb: a backward latency of its own on every boundary;
    every op time against the oracle's evaluation with comm_b."""
    import torch
    for n, seed, mbz in ((61, 3, False), (130, 4, True)):
        batch = W.random_batch(policy, P, M, v, n, seed=seed + P + M, hi=12, comm_hi=6, layout=layout,
                               pad_to=4, stride_mb_zero=mbz)
        cb = np.random.default_rng(seed).integers(0, 9, size=batch.comm.shape).astype(np.int32)
        out = B.evaluate(batch.policy, P, M, v, to_dev(batch.cost_f), to_dev(batch.cost_b), batch.strides, n,
                         comm=to_dev(batch.comm), comm_strides=batch.comm_strides, op_times=True, comm_b=to_dev(cb))
        torch.cuda.synchronize()
        g = {k: t.cpu().numpy() for k, t in out.items()}
        r = orc.eval_batch(batch.policy, P, M, v, batch.cost_f, batch.cost_b, batch.strides, comm=batch.comm,
                           comm_strides=batch.comm_strides, n=n, op_times=True, nthreads=8, comm_b=cb)
        assert_same(g, r, op_times=True)
    # comm_b equal to comm: the same numbers as pp_sched_eval
    same = B.evaluate(batch.policy, P, M, v, to_dev(batch.cost_f), to_dev(batch.cost_b), batch.strides, n,
                      comm=to_dev(batch.comm), comm_strides=batch.comm_strides, comm_b=to_dev(batch.comm))
    base = B.evaluate(batch.policy, P, M, v, to_dev(batch.cost_f), to_dev(batch.cost_b), batch.strides, n,
                      comm=to_dev(batch.comm), comm_strides=batch.comm_strides)
    torch.cuda.synchronize()
    for k in ("makespan", "idle", "bub_num", "bub_den", "status"):
        assert torch.equal(same[k], base[k])


@pytest.mark.parametrize("policy,P,M", [(W.ONEF1B, 8, 16), (W.ONEF1B, 5, 9), (W.GPIPE, 6, 7), (W.GPIPE_FIFO, 8, 5),
                                        (W.ONEF1B, 7, 64)])
def test_two_lanes_per_instance(orc, B, policy, P, M):
    """Small batches of 8-wide GPipe / 1F1B plans without per-op output run
    with two lanes per instance (devices 0-3 and 4-7 exchanging boundary
    arrivals every round): against the oracle, with ragged tails, negative
    costs and overflow."""
    for n, seed in ((1, 1), (17, 2), (250, 3), (1000, 4)):
        batch = W.random_batch(policy, P, M, 1, n, seed=seed * 7 + P + M, hi=30, comm_hi=7, pad_to=4)
        if n >= 250:
            cf = batch.cost_f.reshape(P, M, -1)
            cb = batch.cost_b.reshape(P, M, -1)
            cf[3, M - 1, 5] = -3
            cb[4, 0, 9] = 2**31 - 5
            cf[0, 0, 11] = 2**30
            cb[P - 1, M // 2, 11] = 2**30
        g = run_gpu(batch)
        r = run_oracle(orc, batch)
        assert_same(g, r)
        if n >= 250:
            assert g["status"][5] == B.ST_NEG_COST and g["status"][9] == B.ST_OVERFLOW


@pytest.mark.parametrize("policy,P,M", [(W.ONEF1B, 6, 9), (W.GPIPE, 8, 16), (W.GPIPE_FIFO, 4, 5), (W.ONEF1B, 16, 33)])
@pytest.mark.parametrize("layout", ["inst_minor", "inst_major"])
def test_costs_shared_by_microbatches(orc, B, policy, P, M, layout):
    """stride_mb = 0 (a cost per instance and stage): the register evaluator
    keeps the costs in static round slices; every output against the oracle,
    with and without per-op times, a negative cost and an overflow."""
    for n, seed, ops in ((1, 1, True), (45, 2, False), (300, 3, False), (300, 4, True)):
        batch = W.random_batch(policy, P, M, 1, n, seed=seed + P, hi=40, comm_hi=6, layout=layout,
                               stride_mb_zero=True)
        if n == 300:
            cf = batch.cost_f
            si, ss, _ = batch.strides
            cf[7 * si + 2 * ss] = -1
            batch.cost_b[9 * si + (P - 1) * ss] = 2**31 - 3
        g = run_gpu(batch, op_times=ops)
        r = run_oracle(orc, batch, op_times=ops)
        assert_same(g, r, op_times=ops)
        if n == 300:
            assert g["status"][7] == B.ST_NEG_COST and g["status"][9] == B.ST_OVERFLOW


# Every evaluator kernel writes the plan's peak itself (block 0), so a call is a
# single launch; an empty batch still gets it (a copy on the stream).  Each
# case lands on a different kernel: the one-lane register kernel (inst_minor,
# full and ragged), the microbatch-shared register kernel (stride_mb 0), the
# two-lane 8-wide kernel (small batch, summary outputs), the generic gather
# (instance-major), the lane evaluator (interleaved; GPipe with comm_b).
@pytest.mark.gpu
@pytest.mark.parametrize("policy,P,M,v,n,layout,mbz,comm_b", [
    (W.ONEF1B, 8, 64, 1, 4096, "inst_minor", False, False),
    (W.ONEF1B, 8, 16, 1, 301, "inst_minor", False, False),
    (W.GPIPE, 4, 12, 1, 500, "inst_minor", True, False),
    (W.ONEF1B, 8, 12, 1, 90, "inst_minor", False, False),
    (W.GPIPE_FIFO, 16, 9, 1, 77, "inst_major", False, False),
    (W.INTERLEAVED, 4, 8, 2, 161, "inst_minor", False, False),
    (W.INTERLEAVED, 8, 16, 4, 70, "inst_minor", True, False),
    (W.GPIPE, 4, 8, 1, 33, "inst_major", False, True),
    (W.ONEF1B, 8, 32, 1, 0, "inst_minor", False, False),
])
def test_peak_written_by_every_evaluator(policy, P, M, v, n, layout, mbz, comm_b):
    import torch

    import oracle
    from pipeline_schedule_simulation_gb300 import binding as B
    b = W.random_batch(policy, P, M, v, n, seed=900 + P + M + n, hi=20, layout=layout, stride_mb_zero=mbz)
    out = {"peak": torch.full((P,), -5, dtype=torch.int32, device="cuda")}
    if n:
        out.update(makespan=torch.full((n,), -5, dtype=torch.int32, device="cuda"),
                   status=torch.full((n,), -5, dtype=torch.int8, device="cuda"))
    cm = to_dev(b.comm) if n else None
    B.evaluate(b.policy, P, M, v, to_dev(b.cost_f) if n else torch.zeros(4, dtype=torch.int32, device="cuda"),
               to_dev(b.cost_b) if n else torch.zeros(4, dtype=torch.int32, device="cuda"), b.strides, n,
               comm=cm, comm_strides=b.comm_strides, outputs=("makespan", "peak", "status") if n else ("peak",),
               out=out, comm_b=cm if comm_b else None)
    torch.cuda.synchronize()
    ref = oracle.eval_batch(policy, P, M, v, b.cost_f, b.cost_b, b.strides, comm=b.comm,
                            comm_strides=b.comm_strides, n=n)
    assert np.array_equal(out["peak"].cpu().numpy(), ref["peak"])
    if n:
        assert np.array_equal(out["status"].cpu().numpy(), ref["status"])
        assert np.array_equal(out["makespan"].cpu().numpy(), ref["makespan"])


def test_eval_captured_in_cuda_graph(orc, B):
    """pp_sched_eval once its plan and tables exist launches one kernel and
    allocates nothing, so a CUDA graph can capture it (the benchmark times its
    steps that way): several evaluations captured on a side stream, the graph
    replayed twice after the inputs change in place, every output equal to
    direct calls and to the oracle."""
    import torch
    b = W.hetero_1f1b(n=3001, seed=41)
    cf, cb, cm = to_dev(b.cost_f), to_dev(b.cost_b), to_dev(b.comm)
    out = B.evaluate(b.policy, b.P, b.M, 1, cf, cb, b.strides, b.n, comm=cm, comm_strides=b.comm_strides)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(3):
            B.evaluate(b.policy, b.P, b.M, 1, cf, cb, b.strides, b.n, comm=cm, comm_strides=b.comm_strides, out=out,
                       stream=side)
    for seed in (42, 43):
        nb = W.hetero_1f1b(n=3001, seed=seed)
        cf.copy_(torch.from_numpy(nb.cost_f))
        cb.copy_(torch.from_numpy(nb.cost_b))
        cm.copy_(torch.from_numpy(nb.comm))
        for t in out.values():
            t.fill_(-5)
        graph.replay()
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in out.items()}
        assert_same(got, run_oracle(orc, nb, nthreads=NCPU))


def test_back_to_back_calls_see_previous_outputs(orc, B):
    """Evaluations launched back to back on one stream may overlap their
    starts (programmatic dependent launch); each must still read its inputs
    only after the previous one's writes.  Call 1 writes every op's start and
    end tick (instance-minor, [P*2M][n]); call 2 reads them as its forward and
    backward costs ([S][2M][n], per microbatch, so both calls run the
    one-block-per-SM register kernel).  Three pairs in a row on one stream,
    then the pair captured in a CUDA graph and replayed on new inputs: every
    call 2 equals the oracle run on call 1's times."""
    import torch
    P, M, n = 8, 16, 65536  # enough warps for the one-block-per-SM launch
    O = 2 * M
    b = W.random_batch(W.ONEF1B, P, M, 1, n, seed=21, hi=20, comm_hi=4)
    cf, cb, cm = to_dev(b.cost_f), to_dev(b.cost_b), to_dev(b.comm)
    st = torch.empty(P * O * n, dtype=torch.int32, device="cuda")
    en = torch.empty(P * O * n, dtype=torch.int32, device="cuda")
    out1 = {"op_start": st, "op_end": en}
    s2 = (1, O * n, n)  # call 2: cost of (x, stage k, microbatch j) = time of op j on device k

    def pair(stream):
        B.evaluate(W.ONEF1B, P, M, 1, cf, cb, b.strides, n, comm=cm, comm_strides=b.comm_strides,
                   op_times=True, op_strides=(1, n), out=out1, stream=stream)
        return B.evaluate(W.ONEF1B, P, O, 1, st, en, s2, n, stream=stream)

    def check(o2, shift):
        r1 = orc.eval_batch(W.ONEF1B, P, M, 1, b.cost_f + shift, b.cost_b, b.strides, comm=b.comm,
                            comm_strides=b.comm_strides, n=n, op_times=True, nthreads=16)
        # r1 op times are [n][P][O]: as call 2's costs, strides (P*O, O, 1)
        f2 = r1["op_start"].astype(np.int32).reshape(-1)
        b2 = r1["op_end"].astype(np.int32).reshape(-1)
        r2 = orc.eval_batch(W.ONEF1B, P, O, 1, f2, b2, (P * O, O, 1), n=n, nthreads=16)
        assert_same({k: v.cpu().numpy() for k, v in o2.items()}, r2)

    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for rep in range(3):
            o2 = pair(s)
            outs.append({k: v.clone() for k, v in o2.items()})
            cf.add_(1)  # the next pair's call 1 gets new costs
    torch.cuda.synchronize()
    for rep, o2 in enumerate(outs):
        check(o2, rep)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        o2 = pair(side)
    cf.copy_(to_dev(b.cost_f) + 7)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    check(o2, 7)


def test_back_to_back_costs_shared_by_microbatches(orc, B):
    """Back-to-back calls on the microbatch-shared register kernel: call 1
    (costs per instance and stage, stride_mb 0) writes every op's start and
    end tick; call 2 reads device k's first op start and end as stage k's
    forward and backward cost (stride_mb 0 again), and the next pair's call 1
    rewrites them.  Three pairs on one stream, each call 2 against the oracle
    run on call 1's times."""
    import torch
    P, M, n = 8, 16, 65536
    O = 2 * M
    b = W.random_batch(W.ONEF1B, P, M, 1, n, seed=23, hi=20, comm_hi=4, stride_mb_zero=True)
    assert b.strides[2] == 0 and b.strides[0] == 1
    cf, cb, cm = to_dev(b.cost_f), to_dev(b.cost_b), to_dev(b.comm)
    st = torch.empty(P * O * n, dtype=torch.int32, device="cuda")
    en = torch.empty(P * O * n, dtype=torch.int32, device="cuda")
    out1 = {"op_start": st, "op_end": en}
    s2 = (1, O * n, 0)  # call 2: cost of (x, stage k) = time of op 0 on device k

    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for rep in range(3):
            B.evaluate(W.ONEF1B, P, M, 1, cf, cb, b.strides, n, comm=cm, comm_strides=b.comm_strides,
                       op_times=True, op_strides=(1, n), out=out1, stream=s)
            o2 = B.evaluate(W.ONEF1B, P, M, 1, st, en, s2, n, stream=s)
            outs.append({k: v.clone() for k, v in o2.items()})
            cf.add_(1)
    torch.cuda.synchronize()
    for rep, o2 in enumerate(outs):
        r1 = orc.eval_batch(W.ONEF1B, P, M, 1, b.cost_f + rep, b.cost_b, b.strides, comm=b.comm,
                            comm_strides=b.comm_strides, n=n, op_times=True, nthreads=16)
        f2 = r1["op_start"].astype(np.int32).reshape(-1)  # [n][P][O]
        b2 = r1["op_end"].astype(np.int32).reshape(-1)
        r2 = orc.eval_batch(W.ONEF1B, P, M, 1, f2, b2, (P * O, O, 0), n=n, nthreads=16)
        assert_same({k: v.cpu().numpy() for k, v in o2.items()}, r2)


@pytest.mark.parametrize("P,M,v,n,ops", [(1, 4, 64, 40, True), (2, 4, 32, 70, True), (1, 2, 2, 33, False),
                                         (16, 32, 4, 300, False)])
def test_lane_table_entry_formats(orc, B, P, M, v, n, ops):
    """Interleaved plans whose costs are shared by all microbatches run the
    lane evaluator with one-word table entries while their 2v {cost, comm}
    rows and the zero row fit 7 bits (v = 32 on 2 devices: 65 rows), and the
    cost ring with four-word entries past that (v = 64 on one device: 129
    rows); every output, and every op time where asked, against the oracle."""
    batch = W.random_batch(W.INTERLEAVED, P, M, v, n, seed=5 + P + v, hi=30, comm_hi=6, stride_mb_zero=True)
    assert batch.strides[2] == 0
    g = run_gpu(batch, op_times=ops)
    r = run_oracle(orc, batch, op_times=ops)
    assert (r["status"] == 0).all()
    assert_same(g, r, op_times=ops)


@pytest.mark.parametrize("n,ops", [(4000, True), (12000, False)])
def test_lane_packed_cells_per_cta(orc, B, n, ops):
    """Interleaved, costs shared by all microbatches: a CTA packs its
    {cost, comm} cells into one word when all of its costs and comms lie in
    0 .. 65,535.  One launch where most CTAs pack and a few do not (a cost of
    65,536, a comm of 70,000, a negative cost), with values of exactly 65,535
    in others; one and two instance sets per lane; every output against the
    oracle."""
    P, M, v = 8, 16, 2
    b = W.random_batch(W.INTERLEAVED, P, M, v, n, seed=77 + n, hi=30, comm_hi=6, stride_mb_zero=True)
    si, ss, _ = b.strides
    ci, cbd = b.comm_strides
    b.cost_f[5 * si + 3 * ss] = 65536
    b.cost_b[11 * si + 9 * ss] = 65535
    b.comm[3000 * ci + 4 * cbd] = 70000
    b.comm[3100 * ci + 2 * cbd] = 65535
    b.cost_b[2000 * si + 0 * ss] = -4
    g = run_gpu(b, op_times=ops)
    r = run_oracle(orc, b, op_times=ops)
    assert_same(g, r, op_times=ops)
    assert g["status"][2000] == B.ST_NEG_COST and (np.delete(g["status"], 2000) == 0).all()
