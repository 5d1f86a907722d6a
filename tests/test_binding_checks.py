"""The Python binding refuses buffers the library would address wrongly,
before any library call: tensors on the wrong device, of the wrong dtype, or
shorter than what their element strides reach.  CPU only: every case raises
before a kernel could be launched."""
import numpy as np
import pytest
import torch

from pipeline_schedule_simulation_gb300 import binding as B


def test_reach_counts_the_largest_strided_offset():
    # (n, S, M) = (3, 2, 4), instance-minor strides (1, M*n, n)
    assert B._reach((3, 2, 4), (1, 12, 3)) == 1 + 2 * 1 + 1 * 12 + 3 * 3 == 24
    # a zero stride (costs shared by every microbatch) reaches nothing more
    assert B._reach((3, 2, 4), (2, 1, 0)) == 1 + 2 * 2 + 1
    assert B._reach((0, 2, 4), (1, 12, 3)) == 0
    # brute force on small shapes
    rng = np.random.default_rng(5)
    for _ in range(200):
        ext = tuple(int(x) for x in rng.integers(1, 5, 3))
        st = tuple(int(x) for x in rng.integers(0, 7, 3))
        top = max(a * st[0] + b * st[1] + c * st[2]
                  for a in range(ext[0]) for b in range(ext[1]) for c in range(ext[2]))
        assert B._reach(ext, st) == top + 1


def test_arg_checks_device_dtype_and_length():
    t = torch.zeros(10, dtype=torch.int32)
    assert B._arg(t, "x", torch.int32, None, 10, host=True) is t
    with pytest.raises(ValueError, match="storage holds 10"):
        B._arg(t, "x", torch.int32, None, 11, host=True)
    # a view: the storage counts from the view's data pointer
    with pytest.raises(ValueError, match="storage holds 7"):
        B._arg(t[3:], "x", torch.int32, None, 8, host=True)
    assert B._arg(t[3:5], "x", torch.int32, None, 7, host=True) is not None
    with pytest.raises(TypeError, match="dtype"):
        B._arg(t.to(torch.int64), "x", torch.int32, None, 1, host=True)
    with pytest.raises(ValueError, match="CUDA"):
        B._arg(t, "x", torch.int32, None, 1)
    with pytest.raises(TypeError, match="torch.Tensor"):
        B._arg(np.zeros(4, np.int32), "x", torch.int32, None, 1, host=True)


def test_entry_points_refuse_host_tensors():
    c = torch.ones(4 * 8 * 2, dtype=torch.int32)
    with pytest.raises(ValueError, match="cost_f"):
        B.evaluate(1, 4, 8, 1, c, c, (1, 16, 2), 2)
    with pytest.raises(ValueError, match="cost_f"):
        B.evaluate_zb(3, 4, 8, c, c, c, (1, 16, 2), 2)
    with pytest.raises(ValueError, match="cost_f"):
        B.evaluate_dualpipe(4, 8, 4, c, c, (1, 16, 2), 2)
    with pytest.raises(ValueError, match="layer_tf"):
        B.partition_search(torch.ones(80, dtype=torch.int32), torch.ones(80, dtype=torch.int32),
                           torch.ones(80, dtype=torch.int64), 8, 128, 0, 1 << 40, 1, 0, 16)
    with pytest.raises(ValueError, match="strides"):
        B.evaluate(1, 4, 8, 1, c, c, (1, -16, 2), 2)


def test_host_entry_checks_its_tables():
    n, P, M = 3, 4, 8
    ok = torch.ones(P * M * n, dtype=torch.int32)
    with pytest.raises(ValueError, match="storage holds"):
        B.evaluate_host(1, P, M, 1, ok[1:], ok, n)
    with pytest.raises(TypeError, match="dtype"):
        B.evaluate_host(1, P, M, 1, ok.to(torch.int64), ok, n)
    with pytest.raises(ValueError, match="contiguous"):
        B.evaluate_host(1, P, M, 1, torch.ones(2 * P * M * n, dtype=torch.int32)[::2], ok, n)


@pytest.mark.gpu
def test_short_and_mismatched_device_buffers_are_refused():
    """On the GPU: buffers one element too short for their strides, outputs
    of the wrong dtype or length, and a cost table on another device than the
    others are refused before the library is called; the exact lengths pass."""
    n, P, M = 5, 4, 8
    S = P
    st = (1, M * n, n)  # instance-minor
    need = B._reach((n, S, M), st)
    assert need == n * S * M
    c = torch.ones(need, dtype=torch.int32, device="cuda")
    cm = torch.zeros((S - 1) * n, dtype=torch.int32, device="cuda")
    out = B.evaluate(1, P, M, 1, c, c, st, n, comm=cm, comm_strides=(1, n))
    torch.cuda.synchronize()
    assert (out["status"] == 0).all()
    with pytest.raises(ValueError, match="cost_b"):
        B.evaluate(1, P, M, 1, c, c[1:], st, n)
    with pytest.raises(ValueError, match="comm"):
        B.evaluate(1, P, M, 1, c, c, st, n, comm=cm[1:], comm_strides=(1, n))
    with pytest.raises(TypeError, match="makespan"):
        B.evaluate(1, P, M, 1, c, c, st, n, out={"makespan": torch.empty(n, dtype=torch.int64, device="cuda")})
    with pytest.raises(ValueError, match="idle"):
        B.evaluate(1, P, M, 1, c, c, st, n, out={"idle": torch.empty(n * P - 1, dtype=torch.int32, device="cuda")})
    with pytest.raises(ValueError, match="op_start"):
        B.evaluate(1, P, M, 1, c, c, st, n, op_times=True,
                   out={"op_start": torch.empty(n * P * 2 * M - 1, dtype=torch.int32, device="cuda")})
    with pytest.raises(ValueError, match="cost_w"):
        B.evaluate_zb(3, P, M, c, c, c[2:], st, n)
    with pytest.raises(ValueError, match="cost_b"):
        B.evaluate_dualpipe(P, M, 4, c, c.cpu(), st, n)


def test_binding_api_is_complete():
    """Every public call of the binding is present (a CPU-side guard: most of
    them only run on a GPU)."""
    for name in ("Plan", "op_fields", "evaluate", "evaluate_zb", "evaluate_dualpipe", "evaluate_host", "Many",
                 "partition_search", "partition_search_ranks", "partition_search_interleaved", "cache_clear",
                 "debug_checks", "status_str", "_stream"):
        assert callable(getattr(B, name)), name
