"""Pins of the oracle's DualPipe simulation (orc_dp_inst).

"Pipeline parallelism: from GPipe to 1F1B and Zero Bubble", section "DualPipe
(DeepSeek-V3)": one group of microbatches enters at device 0 and runs the
layer blocks on devices 0..P-1, the other enters at device P-1 and runs the
same blocks on devices P-1..0; each device keeps two blocks (two parameter
copies); a device waiting for one route's input can run the other route's
ready op; the peak of held activations rises from p to p+1.  The page does not
print the merged order; the reading (each route in its own 1F1B order, a free
device runs a ready op of either route, backward before forward, then the
route in which it is the earlier stage) is stated in the oracle.  None of
these tests compares the oracle with itself: each expected value is the 1F1B
oracle (pinned in test_oracle_pins.py), a fact the page states, the bubble of
the comparison table the page shows, a symmetry of the layout, or a separate
tick-by-tick simulation of the reading written here.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore")


def _route_order(P, MA, MB, r, d):
    """Block and ops (kind, global microbatch) of route r on device d, in
    1F1B order: F^w (B F)^(Mr-w) B^w, w = min(P - s, Mr)."""
    s = d if r == 0 else P - 1 - d
    Mr, g0 = (MA, 0) if r == 0 else (MB, MA)
    w = min(P - s, Mr)
    seq = [("F", i) for i in range(w)]
    for q in range(Mr - w):
        seq += [("B", q), ("F", w + q)]
    seq += [("B", i) for i in range(Mr - w, Mr)]
    return s, [(k, g0 + i) for k, i in seq]


def dp_tick_sim(P, MA, MB, tf, tb, comm):
    """The reading simulated one tick at a time: at every tick each free
    device looks at the fronts of its two routes, keeps those whose input has
    arrived, and runs the backward before the forward, then the route in
    which it is the earlier stage.  Returns start and end as [P][2][M]."""
    M = MA + MB
    orders = [[_route_order(P, MA, MB, r, d) for d in range(P)] for r in (0, 1)]
    end, start = {}, {}
    pos = [[0, 0] for _ in range(P)]
    free = [0] * P
    t = 0
    horizon = int(np.sum(tf) + np.sum(tb) + (np.sum(comm) + 1) * 4 * P * M) + 10
    while len(end) < 2 * P * M:
        assert t < horizon
        for d in range(P):
            if free[d] > t:
                continue
            ready = []
            for r in (0, 1):
                s, seq = orders[r][d]
                if pos[d][r] == len(seq):
                    continue
                k, g = seq[pos[d][r]]
                link = (lambda b: b) if r == 0 else (lambda b: P - 2 - b)
                if k == "F":
                    if s == 0:
                        arr = 0
                    else:
                        e = end.get((s - 1, "F", g))
                        arr = None if e is None else e + comm[link(s - 1)]
                else:
                    e0 = end.get((s, "F", g))
                    if s < P - 1:
                        e1 = end.get((s + 1, "B", g))
                        arr = None if e0 is None or e1 is None else max(e0, e1 + comm[link(s)])
                    else:
                        arr = e0
                if arr is not None and arr <= t:
                    ready.append((k == "F", r != (0 if d <= P - 1 - d else 1), r, k, g, s))
            if not ready:
                continue
            _, _, r, k, g, s = min(ready)
            c = int(tf[s][g] if k == "F" else tb[s][g])
            start[(s, k, g)], end[(s, k, g)] = t, t + c
            free[d] = t + c
            pos[d][r] += 1
        t += 1
    S = np.zeros((P, 2, M), np.int64)
    E = np.zeros((P, 2, M), np.int64)
    for (s, k, g), v in start.items():
        S[s, 0 if k == "F" else 1, g] = v
        E[s, 0 if k == "F" else 1, g] = end[(s, k, g)]
    return S, E


def test_one_route_alone_is_1f1b(orc):
    """With the other route empty, each route is plain 1F1B on its P devices:
    route A on devices 0..P-1 with the links in order, route B on devices
    P-1..0, whose boundary b is link P-2-b."""
    rng = np.random.default_rng(1)
    for P in (1, 2, 3, 4, 7, 8):
        for M in (1, 2, 5, 9, 16):
            tf = rng.integers(1, 9, size=(P, M))
            tb = rng.integers(1, 9, size=(P, M))
            cm = rng.integers(0, 4, size=max(P - 1, 1))
            a = orc.dp_evaluate(P, M, 0, tf, tb, cm)
            r = orc.evaluate("1f1b", P, M, 1, tf, tb, cm)
            # the 1F1B oracle's times are by device and position; map them to (block, kind, microbatch)
            for k in range(P):
                for j in range(2 * M):
                    kd, mb = r["kind"][k, j], r["mb"][k, j]
                    assert a["start"][k, kd, mb] == r["start"][k, j]
            assert a["makespan"] == r["makespan"] and list(a["peak"]) == list(r["peak"])
            b = orc.dp_evaluate(P, 0, M, tf, tb, cm)
            rb = orc.evaluate("1f1b", P, M, 1, tf, tb, cm[::-1].copy() if P > 1 else cm)
            for s in range(P):
                for j in range(2 * M):
                    kd, mb = rb["kind"][s, j], rb["mb"][s, j]
                    assert b["start"][s, kd, mb] == rb["start"][s, j]
            # route B's block s runs on device P-1-s
            assert list(b["peak"]) == list(rb["peak"])[::-1]
            assert b["makespan"] == rb["makespan"]


def test_two_blocks_per_device_and_the_page_peak(orc):
    """Each device runs route A's block d and route B's block P-1-d (its busy
    time is exactly those ops' costs: two copies of the parameters), and holds
    at most P+1 activations; with at least P microbatches on each route the
    peak is P+1, one more than 1F1B's P, as the page states."""
    rng = np.random.default_rng(2)
    for P in (2, 3, 4, 6, 8, 16):
        for MA, MB in ((1, 1), (P, P), (P + 3, P), (2 * P, 2 * P + 1), (3, 2 * P)):
            M = MA + MB
            for uniform in (True, False):
                tf = np.full((P, M), 2) if uniform else rng.integers(1, 9, size=(P, M))
                tb = np.full((P, M), 3) if uniform else rng.integers(1, 9, size=(P, M))
                cm = np.zeros(max(P - 1, 1), np.int64) if uniform else rng.integers(0, 4, size=max(P - 1, 1))
                r = orc.dp_evaluate(P, MA, MB, tf, tb, cm)
                for d in range(P):
                    want = tf[d, :MA].sum() + tb[d, :MA].sum() + tf[P - 1 - d, MA:].sum() + tb[P - 1 - d, MA:].sum()
                    assert r["busy"][d] == want
                    # each route's own ledger peaks at min(P - stage, Mr) under 1F1B
                    assert r["peak"][d] <= min(P - d, MA) + min(d + 1, MB) <= P + 1
                if MA >= P and MB >= P and uniform:
                    assert max(r["peak"]) == P + 1


def test_uniform_bubble_matches_comparison_table(orc):
    """The comparison table the page shows (DeepSeek-V3's) gives DualPipe's
    bubble as (PP/2 - 1)(F&B + B - 3W), against (PP - 1)(F + B) for 1F1B.
    Here a forward and a backward do not overlap (F&B = F + B) and the weight
    gradient is not split off (W = 0), so each device idles (P/2 - 1)(t_f +
    2 t_b) ticks at uniform costs, for t_b >= t_f (the pages' workloads have
    t_b about 2 t_f), even P and at least P microbatches per route."""
    for tf, tb in ((1, 1), (1, 2), (2, 3), (3, 5), (2, 4)):
        for P in (2, 4, 6, 8, 16):
            for M in (2 * P, 3 * P, 4 * P + 2, 8 * P):
                MA = (M + 1) // 2
                r = orc.dp_evaluate(P, MA, M - MA, tf, tb)
                idle = (P // 2 - 1) * (tf + 2 * tb)
                assert list(r["idle"]) == [idle] * P, (tf, tb, P, M)
                assert r["makespan"] == M * (tf + tb) + idle
                # against the 1F1B row of the same table, (P - 1)(t_f + t_b) per device
                assert idle <= (P - 1) * (tf + tb)


def test_mirror_symmetry(orc):
    """Mirroring the devices (d -> P-1-d) swaps the routes.  With equal route
    sizes, the same costs for route A's i-th and route B's i-th microbatch and
    a link latency equal to its mirror's, route B's times equal route A's, and
    the device peaks read the same backwards (P even, where no device is the
    same stage on both routes)."""
    rng = np.random.default_rng(3)
    for P in (2, 4, 6, 8):
        for MA in (1, 3, P, 2 * P + 1):
            half_f = rng.integers(1, 9, size=(P, MA))
            half_b = rng.integers(1, 9, size=(P, MA))
            tf = np.concatenate([half_f, half_f], axis=1)
            tb = np.concatenate([half_b, half_b], axis=1)
            c = rng.integers(0, 4, size=max(P - 1, 1))
            cm = np.minimum(c, c[::-1])
            r = orc.dp_evaluate(P, MA, MA, tf, tb, cm)
            assert np.array_equal(r["start"][:, :, :MA], r["start"][:, :, MA:])
            assert list(r["peak"]) == list(r["peak"])[::-1]


def test_tick_simulation_agrees(orc):
    """A separate tick-by-tick simulation of the reading gives every op's
    start and end."""
    rng = np.random.default_rng(4)
    for _ in range(250):
        P = int(rng.integers(1, 7))
        MA = int(rng.integers(0, 7))
        MB = int(rng.integers(0 if MA else 1, 7))
        M = MA + MB
        tf = rng.integers(1, 6, size=(P, M))
        tb = rng.integers(1, 6, size=(P, M))
        cm = rng.integers(0, 4, size=max(P - 1, 1))
        r = orc.dp_evaluate(P, MA, MB, tf, tb, cm)
        S, E = dp_tick_sim(P, MA, MB, tf, tb, cm)
        assert np.array_equal(r["start"], S), (P, MA, MB)
        assert np.array_equal(r["end"], E)


def test_batch_statuses(orc):
    """The batch form: strides, negative and zero costs, overflow."""
    P, MA, MB, n = 4, 3, 2, 6
    M = MA + MB
    rng = np.random.default_rng(5)
    cf = rng.integers(1, 9, size=(n, P, M)).astype(np.int32)
    cb = rng.integers(1, 9, size=(n, P, M)).astype(np.int32)
    cm = rng.integers(0, 4, size=(n, P - 1)).astype(np.int32)
    cf[1, 2, 3] = -1
    cb[2, 0, 0] = 0
    cm[3, 1] = -2
    cb[4, 1, 1] = 2**31 - 5
    out = orc.dp_batch(P, MA, MB, cf.reshape(-1), cb.reshape(-1), (P * M, M, 1), cm.reshape(-1), (P - 1, 1), n=n,
                       op_times=True)
    assert list(out["status"]) == [0, orc.ST_NEG_COST, orc.ST_ZERO_COST, orc.ST_NEG_COST, orc.ST_OVERFLOW, 0]
    for x in (0, 5):
        r = orc.dp_evaluate(P, MA, MB, cf[x], cb[x], cm[x])
        assert out["makespan"][x] == r["makespan"]
        assert np.array_equal(out["op_start"][x], r["start"])
        assert np.array_equal(out["peak"][x], r["peak"])
