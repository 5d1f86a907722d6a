"""The seeded generators draw what the workloads state (ranges, shapes, seeds)."""
import numpy as np

import pipeline_schedule_simulation_gb300.workloads as W


def test_hetero_1f1b_ranges_and_determinism():
    a = W.hetero_1f1b(n=2048)
    b = W.hetero_1f1b(n=2048)
    assert np.array_equal(a.cost_f, b.cost_f) and np.array_equal(a.comm, b.comm)
    assert a.cost_f.min() >= 80 and a.cost_f.max() <= 120
    assert a.cost_b.min() >= 160 and a.cost_b.max() <= 240
    assert a.comm.min() >= 2 and a.comm.max() <= 8
    assert a.cost_f.size == 8 * 64 * 2048 and a.strides == (1, 64 * 2048, 2048)
    # inclusive ranges: the end points occur
    assert a.cost_f.max() == 120 and a.comm.max() == 8


def test_interleaved_equal_work():
    il, base = W.interleaved_vs_1f1b(2, n=512)
    tf = il.cost_f.reshape(16, 512)
    assert tf.min() >= 40 and tf.max() <= 60
    tb = il.cost_b.reshape(16, 512)
    assert np.all(np.abs(tb - 2 * tf) <= 5)
    assert np.array_equal(base.cost_f.reshape(8, 512), tf[:8] + tf[8:])
    assert il.strides == (1, 512, 0)


def test_layer_split_layers():
    p = W.layer_split()
    assert p.layer_tf.shape == (80,)
    assert 135 <= p.layer_tf[0] <= 165 and 270 <= p.layer_tf[79] <= 330
    assert np.all((p.layer_tf[1:79] >= 90) & (p.layer_tf[1:79] <= 110))
    assert np.array_equal(p.layer_tb, 2 * p.layer_tf)
    assert p.layer_act.min() >= 200 * 10**6 and p.layer_act.max() <= 300 * 10**6
    assert p.cap == 80 * 10**9 and p.n_cand == 1 << 20


def test_sweep_shapes():
    shapes = W.sweep_shapes()
    assert len([s for s in shapes if s[0] == W.GPIPE]) == 15 * 128
    il = [s for s in shapes if s[0] == W.INTERLEAVED]
    assert all(M % P == 0 and v == 2 for _, P, M, v in il)
    b = W.sweep_batch(W.ONEF1B, 4, 8, 1)
    assert b.n == 16 and b.strides == (1, 0, 0)
