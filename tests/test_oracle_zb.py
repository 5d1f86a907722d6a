"""Pins of the oracle's Zero Bubble schedules (ZB1P, ZB2P), without a GPU.

The rules ("Pipeline parallelism: from GPipe to 1F1B and Zero Bubble",
sections "Zero Bubble" and "ZB1P and ZB2P"): the backward splits into B (input
gradient, needed by the previous stage) and W (weight gradient, no
cross-stage edge); 1F1B's F/B order is kept and a gap where the next F/B's
input has not arrived is filled with a ready W; a device holds at most P
(ZB1P) or 2P (ZB2P) microbatches whose W has not run.  The pages print no
timeline, so the pins are: worked examples derived by hand from the rules
(tests/golden/zb*_p2m2_unit.txt), the reduction to schedules pinned
elsewhere when W costs nothing, and an independent tick-stepped simulation of
the same rules.
"""
import numpy as np
import pytest

from conftest import read_golden

KIND = {"F": 0, "B": 1, "W": 2}


def _timeline(r, P, M, span):
    """Unit-cost rows: the op occupying each tick of each device."""
    rows = []
    for k in range(P):
        row = ["-"] * span
        for name, kd in KIND.items():
            for m in range(M):
                row[r["start"][k, kd, m]] = f"{name}{m}"
        rows.append(row)
    return rows


@pytest.mark.parametrize("policy,fixture", [("zb1p", "zb1p_p2m2_unit.txt"), ("zb2p", "zb2p_p2m2_unit.txt")])
def test_zb_worked_examples(orc, policy, fixture):
    g = read_golden(fixture)
    r = orc.zb_evaluate(policy, 2, 2, 1, 1, 1)
    span = int(g["makespan"][0])
    assert r["makespan"] == span
    assert _timeline(r, 2, 2, span) == [g["stage0"], g["stage1"]]
    assert r["bub"] == tuple(int(x) for x in g["bubble"])
    assert list(r["peak"]) == [int(x) for x in g["peak"]]


def zb_tick_sim(policy, P, M, tf, tb, tw, comm):
    """The ZB rules run tick by tick: at every tick each free device, in index
    order, takes the first rule that applies (a W of zero cost lets it decide
    again at the same tick).  Returns start/end [P][3][M] and the peaks."""
    L = P if policy == "zb1p" else 2 * P
    seqs = []
    for k in range(P):
        w = min(P - k if policy == "zb1p" else 2 * (P - k), M)
        seq = [("F", i) for i in range(w)]
        for q in range(M - w):
            seq += [("B", q), ("F", w + q)]
        seq += [("B", i) for i in range(M - w, M)]
        seqs.append(seq)
    cost = {"F": tf, "B": tb, "W": tw}
    start, end = {}, {}
    free, pos, held, peak = [0] * P, [0] * P, [0] * P, [0] * P
    pending = [[] for _ in range(P)]

    def arrival(k, kd, m):
        if kd == "F":
            if k == 0:
                return 0
            e = end.get((k - 1, "F", m))
            return None if e is None else e + comm[k - 1]
        if k == P - 1:
            return end[(k, "F", m)]
        e = end.get((k + 1, "B", m))
        return None if e is None else e + comm[k]

    t = 0
    while len(end) < 3 * P * M:
        assert t < 10**6
        for k in range(P):
            while free[k] <= t:
                run = None
                if pos[k] < 2 * M:
                    kd, m = seqs[k][pos[k]]
                    a = arrival(k, kd, m)
                    if kd == "F" and held[k] >= L:
                        run = ("W", pending[k][0])
                    elif a is not None and a <= t:
                        run = (kd, m)
                    elif pending[k]:
                        run = ("W", pending[k][0])
                elif pending[k]:
                    run = ("W", pending[k][0])
                if run is None:
                    break
                kd, m = run
                start[(k, kd, m)] = t
                end[(k, kd, m)] = t + int(cost[kd][k][m])
                free[k] = end[(k, kd, m)]
                if kd == "W":
                    pending[k].pop(0)
                    held[k] -= 1
                else:
                    pos[k] += 1
                    if kd == "F":
                        held[k] += 1
                        peak[k] = max(peak[k], held[k])
                    else:
                        pending[k].append(m)
        t += 1
    S = np.zeros((P, 3, M), np.int64)
    E = np.zeros((P, 3, M), np.int64)
    for (k, kd, m), v in start.items():
        S[k, KIND[kd], m] = v
        E[k, KIND[kd], m] = end[(k, kd, m)]
    return S, E, peak


def _random_case(rng, P, M, w_lo=0):
    tf = rng.integers(1, 6, size=(P, M))
    tb = rng.integers(1, 6, size=(P, M))
    tw = rng.integers(w_lo, 5, size=(P, M))
    comm = rng.integers(0, 4, size=max(P - 1, 1))
    return tf, tb, tw, comm


@pytest.mark.parametrize("policy", ["zb1p", "zb2p"])
def test_zb_matches_tick_simulation(orc, policy):
    rng = np.random.default_rng(7 if policy == "zb1p" else 8)
    for P in range(1, 6):
        for M in (1, 2, 3, 5, 8):
            for _ in range(6):
                tf, tb, tw, comm = _random_case(rng, P, M)
                r = orc.zb_evaluate(policy, P, M, tf, tb, tw, comm)
                S, E, peak = zb_tick_sim(policy, P, M, tf, tb, tw, comm)
                assert np.array_equal(r["start"], S), (policy, P, M)
                assert np.array_equal(r["end"], E)
                assert list(r["peak"]) == peak
                assert r["makespan"] == E.max()


def test_zb1p_without_w_is_1f1b(orc):
    """With every W free, ZB1P's F and B run exactly as 1F1B's F and B."""
    rng = np.random.default_rng(11)
    for P, M in ((1, 4), (2, 2), (3, 7), (4, 8), (6, 5), (8, 16)):
        for _ in range(4):
            tf, tb, _, comm = _random_case(rng, P, M)
            r = orc.zb_evaluate("zb1p", P, M, tf, tb, 0, comm)
            ref = orc.evaluate("1f1b", P, M, 1, tf, tb, comm)
            for k in range(P):
                for j in range(2 * M):
                    kd, m = ref["kind"][k, j], ref["mb"][k, j]
                    assert r["start"][k, kd, m] == ref["start"][k, j]
                    assert r["end"][k, kd, m] == ref["end"][k, j]
            assert r["makespan"] == ref["makespan"]


def test_zb2p_without_w_is_its_explicit_order(orc):
    """With every W free, ZB2P's F and B follow the explicit order with the
    doubled warmup, evaluated by the oracle's event simulation and longest
    path (pinned by the 1F1B / GPipe tests)."""
    rng = np.random.default_rng(12)
    for P, M in ((2, 2), (3, 9), (4, 6), (5, 12)):
        for _ in range(4):
            tf, tb, _, comm = _random_case(rng, P, M)
            kind = np.zeros((P, 2 * M), np.int32)
            mb = np.zeros((P, 2 * M), np.int32)
            for k in range(P):
                w = min(2 * (P - k), M)
                seq = [(0, i) for i in range(w)]
                for q in range(M - w):
                    seq += [(1, q), (0, w + q)]
                seq += [(1, i) for i in range(M - w, M)]
                kind[k] = [a for a, _ in seq]
                mb[k] = [b for _, b in seq]
            ref = orc.eval_explicit(P, M, 1, kind, np.zeros_like(kind), mb, tf, tb, comm)
            r = orc.zb_evaluate("zb2p", P, M, tf, tb, 0, comm)
            for k in range(P):
                for j in range(2 * M):
                    assert r["start"][k, kind[k, j], mb[k, j]] == ref["start"][k, j]
            assert r["makespan"] == ref["makespan"]


def test_zb_budget_and_counts(orc):
    """Peaks stay within P (ZB1P) or 2P (ZB2P) even when W dominates; busy
    time is every op's cost; idle and bubble follow the window definition."""
    rng = np.random.default_rng(13)
    for policy, L in (("zb1p", 1), ("zb2p", 2)):
        for P, M in ((2, 6), (3, 12), (4, 16)):
            tf = rng.integers(1, 4, size=(P, M))
            tb = rng.integers(1, 4, size=(P, M))
            tw = rng.integers(8, 20, size=(P, M))
            r = orc.zb_evaluate(policy, P, M, tf, tb, tw, np.ones(P - 1, np.int64))
            assert (r["peak"] <= L * P).all()
            assert r["peak"][0] == min(L * P, M)
            assert np.array_equal(r["busy"], (tf + tb + tw).sum(axis=1))
            assert np.array_equal(r["idle"], r["makespan"] - r["busy"])
            assert r["bub"] == (int(r["idle"].sum()), P * r["makespan"])


def test_zb_fills_1f1b_bubble(orc):
    """W placed in the gaps: with F = B = W = 1 tick and no comm, ZB1P ends
    before 1F1B with the same total backward (B + W = 2 ticks) whenever
    there is more than one device."""
    for P in range(2, 7):
        for M in (P, 2 * P, 3 * P):
            zb = orc.zb_evaluate("zb1p", P, M, 1, 1, 1)
            f1 = orc.evaluate("1f1b", P, M, 1, 1, 2)
            assert zb["makespan"] < f1["makespan"] == (M + P - 1) * 3


def test_zb_rejects_costs_below_one(orc):
    with pytest.raises(orc.OracleError):
        orc.zb_evaluate("zb1p", 2, 2, 1, 0, 1)
    out = orc.zb_batch("zb1p", 2, 2, np.array([1, 0, 1, 1, 1, 1, 1, 1], np.int32),
                       np.ones(8, np.int32), np.zeros(8, np.int32), (4, 2, 1),
                       comm=np.array([0, -1], np.int32), comm_strides=(1, 0), n=2)
    # instance 0: an F of zero cost; instance 1: a negative comm (W may be 0)
    assert list(out["status"]) == [orc.ST_ZERO_COST, orc.ST_NEG_COST]


def test_zb_batch_matches_single(orc):
    rng = np.random.default_rng(14)
    P, M, n = 4, 6, 9
    cf = rng.integers(1, 9, size=(n, P, M)).astype(np.int32)
    cb = rng.integers(1, 9, size=(n, P, M)).astype(np.int32)
    cw = rng.integers(0, 9, size=(n, P, M)).astype(np.int32)
    cm = rng.integers(0, 3, size=(n, P - 1)).astype(np.int32)
    for policy in ("zb1p", "zb2p"):
        out = orc.zb_batch(policy, P, M, cf.reshape(-1), cb.reshape(-1), cw.reshape(-1), (P * M, M, 1),
                           comm=cm.reshape(-1), comm_strides=(P - 1, 1), n=n, op_times=True, nthreads=3)
        for x in range(n):
            r = orc.zb_evaluate(policy, P, M, cf[x], cb[x], cw[x], cm[x])
            assert out["makespan"][x] == r["makespan"] and out["status"][x] == 0
            assert np.array_equal(out["idle"][x], r["idle"])
            assert np.array_equal(out["peak"][x], r["peak"])
            assert (out["bub_num"][x], out["bub_den"][x]) == r["bub"]
            assert np.array_equal(out["op_start"][x], r["start"])
            assert np.array_equal(out["op_end"][x], r["end"])
