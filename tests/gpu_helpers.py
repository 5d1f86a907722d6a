"""Shared helpers of the GPU parity tests: run a workload Batch through the
library (C ABI via the binding) and through the oracle, on the same inputs."""
import numpy as np
import torch


def to_dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gpu(batch, op_times=False):
    from pipeline_schedule_simulation_gb300 import binding as B
    out = B.evaluate(batch.policy, batch.P, batch.M, batch.v, to_dev(batch.cost_f), to_dev(batch.cost_b),
                     batch.strides, batch.n, comm=to_dev(batch.comm), comm_strides=batch.comm_strides,
                     op_times=op_times)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_oracle(orc, batch, op_times=False, nthreads=8, select=None):
    """Oracle outputs for all instances, or for the instance indices in `select`."""
    if select is None:
        return orc.eval_batch(batch.policy, batch.P, batch.M, batch.v, batch.cost_f, batch.cost_b,
                              batch.strides, comm=batch.comm, comm_strides=batch.comm_strides,
                              n=batch.n, op_times=op_times, nthreads=nthreads)
    # gather the selected instances into a small instance-major batch
    S, M = batch.S, batch.M
    si, ss, sm = batch.strides
    idx = np.asarray(select, np.int64)
    s_ix = np.arange(S)[None, :, None]
    m_ix = np.arange(M)[None, None, :]
    off = idx[:, None, None] * si + s_ix * ss + m_ix * sm
    cf = batch.cost_f[off].astype(np.int32)
    cb = batch.cost_b[off].astype(np.int32)
    cm = None
    if batch.comm is not None:
        ci, cbd = batch.comm_strides
        cm = batch.comm[idx[:, None] * ci + np.arange(max(S - 1, 1))[None, :] * cbd].astype(np.int32)
    return orc.eval_batch(batch.policy, batch.P, batch.M, batch.v, cf, cb, (S * M, M, 1), comm=cm,
                          comm_strides=(max(S - 1, 1), 1), n=len(idx), op_times=op_times,
                          nthreads=nthreads)


def assert_same(gpu, ref, select=None, op_times=False):
    ok = ref["status"] == 0
    g = {k: (v if select is None or k == "peak" else v[np.asarray(select)]) for k, v in gpu.items()}
    assert np.array_equal(g["status"], ref["status"])
    assert np.array_equal(g["peak"], ref["peak"])
    assert np.array_equal(g["makespan"][ok], ref["makespan"][ok])
    assert np.array_equal(g["idle"][ok], ref["idle"][ok])
    assert np.array_equal(g["bub_num"][ok], ref["bub_num"][ok])
    assert np.array_equal(g["bub_den"][ok], ref["bub_den"][ok])
    # the float view of the bubble agrees far inside 1e-12
    den = np.maximum(ref["bub_den"][ok], 1)
    assert np.all(np.abs(g["bub_num"][ok] / np.maximum(g["bub_den"][ok], 1) - ref["bub_num"][ok] / den) <= 1e-12)
    if op_times:
        assert np.array_equal(g["op_start"][ok], ref["op_start"][ok])
        assert np.array_equal(g["op_end"][ok], ref["op_end"][ok])


def run_gpu_zb(batch, op_times=False):
    from pipeline_schedule_simulation_gb300 import binding as B
    out = B.evaluate_zb(batch.policy, batch.P, batch.M, to_dev(batch.cost_f), to_dev(batch.cost_b),
                        to_dev(batch.cost_w), batch.strides, batch.n, comm=to_dev(batch.comm),
                        comm_strides=batch.comm_strides, op_times=op_times)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_oracle_zb(orc, batch, op_times=False, nthreads=8, select=None):
    """Oracle outputs of a Zero Bubble batch, for all instances or `select`."""
    if select is None:
        return orc.zb_batch(batch.policy, batch.P, batch.M, batch.cost_f, batch.cost_b, batch.cost_w,
                            batch.strides, comm=batch.comm, comm_strides=batch.comm_strides, n=batch.n,
                            op_times=op_times, nthreads=nthreads)
    P, M = batch.P, batch.M
    si, ss, sm = batch.strides
    idx = np.asarray(select, np.int64)
    off = idx[:, None, None] * si + np.arange(P)[None, :, None] * ss + np.arange(M)[None, None, :] * sm
    ci, cbd = batch.comm_strides
    cm = batch.comm[idx[:, None] * ci + np.arange(max(P - 1, 1))[None, :] * cbd].astype(np.int32)
    return orc.zb_batch(batch.policy, P, M, batch.cost_f[off].astype(np.int32), batch.cost_b[off].astype(np.int32),
                        batch.cost_w[off].astype(np.int32), (P * M, M, 1), comm=cm,
                        comm_strides=(max(P - 1, 1), 1), n=len(idx), op_times=op_times, nthreads=nthreads)


def assert_same_zb(gpu, ref, select=None, op_times=False):
    ok = ref["status"] == 0
    g = {k: (v if select is None else v[np.asarray(select)]) for k, v in gpu.items()}
    assert np.array_equal(g["status"], ref["status"])
    for key in ("makespan", "idle", "bub_num", "bub_den", "peak"):
        assert np.array_equal(g[key][ok], ref[key][ok]), key
    if op_times:
        assert np.array_equal(g["op_start"][ok], ref["op_start"][ok])
        assert np.array_equal(g["op_end"][ok], ref["op_end"][ok])


def run_gpu_dp(batch, m_a, op_times=False):
    from pipeline_schedule_simulation_gb300 import binding as B
    out = B.evaluate_dualpipe(batch.P, batch.M, m_a, to_dev(batch.cost_f), to_dev(batch.cost_b), batch.strides,
                              batch.n, comm=to_dev(batch.comm), comm_strides=batch.comm_strides, op_times=op_times)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_oracle_dp(orc, batch, m_a, op_times=False, nthreads=8):
    return orc.dp_batch(batch.P, m_a, batch.M - m_a, batch.cost_f, batch.cost_b, batch.strides, comm=batch.comm,
                        comm_strides=batch.comm_strides, n=batch.n, op_times=op_times, nthreads=nthreads)
