"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compare the oracle with itself: each expected value is a cell of
a table the pages print, a closed form the pages state, a brute-force optimum,
a published test vector, or a library routine (math.comb, itertools).
"""
import itertools
import math
import os
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore")


def _table_from_oracle(r, P, names="ABCD"):
    rows = []
    for k in range(P):
        row = ["-"] * r["makespan"]
        for j in range(r["kind"].shape[1]):
            kd = "F" if r["kind"][k, j] == 0 else "B"
            row[r["start"][k, j]] = f"{kd}-{names[r['mb'][k, j]]}"
        rows.append(row)
    return rows


@pytest.mark.parametrize("policy,fixture", [("gpipe", "m040_gpipe_2x4.txt"), ("1f1b", "m040_1f1b_2x4.txt")])
def test_m040_worked_tables_cell_for_cell(orc, policy, fixture):
    g = read_golden(fixture)
    r = orc.evaluate(policy, 2, 4, 1, 1, 1)
    assert _table_from_oracle(r, 2) == [g["stage0"], g["stage1"]]
    assert r["makespan"] == int(g["window"][0])
    assert r["peak"][0] == int(g["peak_stage0"][0])
    if "busy_percent" in g:
        num, den = r["bub"]
        assert Fraction(den - num, den) == Fraction(int(g["busy_percent"][0]), 100)


def test_onef1b_p4m6_diagram_and_ledger(orc):
    g = read_golden("onef1b_p4m6.txt")
    r = orc.evaluate("1f1b", 4, 6, 1, 1, 1)
    k0 = [f"{'FB'[r['kind'][0, j]]}{r['mb'][0, j]}" for j in range(12)]
    assert k0 == g["stage0_order"]
    k3 = [f"{'FB'[r['kind'][3, j]]}{r['mb'][3, j]}" for j in range(12)]
    assert k3 == g["stage3_order"]
    times = dict(x.split("=") for x in g["stage0_time"])
    for j, name in enumerate(k0):
        if name in times:
            assert r["start"][0, j] == int(times[name]), name
    held, ledger = 0, []
    for j in range(12):
        held += 1 if r["kind"][0, j] == 0 else -1
        ledger.append(held)
    assert ledger == [int(x) for x in g["stage0_ledger"]]
    assert r["peak"][0] == int(g["stage0_peak"][0])


@pytest.mark.parametrize("policy", ["gpipe", "1f1b"])
def test_uniform_closed_form(orc, policy):
    # "2. 1F1B" §4.3 and M040 §04: total 2(M+P-1)tau, busy M/(M+P-1),
    # bubble (P-1)/(M+P-1), identical for GPipe and 1F1B.
    for P in range(1, 9):
        for M in list(range(1, 13)) + [17, 24]:
            for tau in (1, 3):
                r = orc.evaluate(policy, P, M, 1, tau, tau, method=2)
                assert r["makespan"] == 2 * (M + P - 1) * tau
                num, den = r["bub"]
                assert Fraction(num, den) == Fraction(P - 1, M + P - 1)
                assert all(r["busy"] == 2 * M * tau)


@pytest.mark.parametrize("policy", ["gpipe", "1f1b"])
def test_tf_tb_closed_form(orc, policy):
    # "From GPipe to 1F1B and Zero Bubble", Megatron section: bubble overhead
    # (p-1)(t_f+t_b) on top of the ideal m(t_f+t_b); PipeDream-Flush has the same
    # bubble.  So total = (m+p-1)(t_f+t_b), e.g. t_b = 2 t_f ("lpnh" article).
    for P in range(1, 9):
        for M in (1, 2, 5, 8, 13, 24):
            for tf, tb in ((1, 2), (2, 4), (3, 1), (2, 5)):
                r = orc.evaluate(policy, P, M, 1, tf, tb, method=2)
                assert r["makespan"] == (M + P - 1) * (tf + tb)


def test_lpnh_30_4_percent(orc):
    # lpnh article: P = 8, M = 16 gives a 30.4 % bubble for GPipe.
    for policy in ("gpipe", "1f1b"):
        num, den = orc.evaluate(policy, 8, 16, 1, 1, 1)["bub"]
        assert Fraction(num, den) == Fraction(7, 23)
        assert round(100 * num / den, 1) == 30.4


def test_p4_m8_tf1_tb2_values(orc):
    # P=4, M=8, t_f=1, t_b=2: (M+P-1)(t_f+t_b) = 33, busy 24 per stage, bubble 3/11.
    for policy in ("gpipe", "1f1b"):
        r = orc.evaluate(policy, 4, 8, 1, 1, 2, method=2)
        assert r["makespan"] == 33
        assert list(r["busy"]) == [24] * 4
        assert list(r["idle"]) == [9] * 4
        assert r["bub"] == (36, 132)
    assert list(orc.evaluate("gpipe", 4, 8, 1, 1, 2)["peak"]) == [8, 8, 8, 8]
    assert list(orc.evaluate("1f1b", 4, 8, 1, 1, 2)["peak"]) == [4, 3, 2, 1]


def test_1f1b_phases_and_warmup_conventions(orc):
    # "2. 1F1B" §2.3/§3.2: stage k runs P-k forwards before its first B, then
    # M-(P-k) F-B pairs, then P-k backwards.  "Megatron-LM (3)": num_warmup =
    # P-k-1, then the steady phase starts with a forward; same count.
    for P in range(1, 9):
        for M in range(1, 20):
            kind, _, mb = orc.order("1f1b", P, M)
            for k in range(P):
                seq = list(kind[k])
                first_b = seq.index(1)
                assert first_b == min(P - k, M)
                megatron_warmup = min(P - k - 1, M)
                if M > P - k - 1:
                    assert seq[megatron_warmup] == 0  # steady phase opens with F
                if M >= P - k:
                    w = P - k
                    steady = seq[w:w + 2 * (M - w)]
                    assert steady == [1, 0] * (M - w)
                    assert seq[w + 2 * (M - w):] == [1] * w
                # oldest outstanding microbatch first
                bs = [mb[k, j] for j in range(2 * M) if kind[k, j] == 1]
                assert bs == list(range(M))


def test_peaks(orc):
    # "2. 1F1B" §4.1/§4.5: 1F1B holds P on stage 0 whatever M is; GPipe holds M.
    for P in range(1, 9):
        for M in (1, 2, 3, 6, 60, 100):
            p1 = orc.evaluate("1f1b", P, M, 1, 1, 1)["peak"]
            assert list(p1) == [min(P - k, M) for k in range(P)]
            assert max(p1) <= P
            pg = orc.evaluate("gpipe", P, M, 1, 1, 1)["peak"]
            assert list(pg) == [M] * P


def test_interleaved_bubble_and_divisibility(orc):
    # "2. 1F1B" §6.1: bubble (P-1)/(V*M+P-1) for interleaved 1F1B.
    for P in (1, 2, 3, 4, 8):
        for v in (2, 3, 4):
            for M in (P, 2 * P, 4 * P):
                r = orc.evaluate("interleaved", P, M, v, 1, 1, method=2)
                num, den = r["bub"]
                assert Fraction(num, den) == Fraction(P - 1, v * M + P - 1)
    num, den = orc.evaluate("interleaved", 8, 128, 4, 1, 1)["bub"]
    assert Fraction(num, den) == Fraction(7, 519)
    # M040 §06: frameworks may require divisibility; M % P != 0 is refused.
    with pytest.raises(orc.OracleError) as e:
        orc.order("interleaved", 4, 6, 2)
    assert e.value.code == orc.ERR_DIVISIBILITY


def test_interleaved_placement(orc):
    # "From GPipe to 1F1B and Zero Bubble", Megatron section; M040 §06: device k
    # holds virtual stages k, k+P, ...; every device runs each chunk's M F and M B.
    P, M, v = 4, 8, 2
    kind, chunk, mb = orc.order("interleaved", P, M, v)
    for k in range(P):
        for c in range(v):
            for kd in (0, 1):
                sel = (kind[k] == kd) & (chunk[k] == c)
                assert sorted(mb[k][sel]) == list(range(M))


def test_interleaved_warmup_from_first_gradient(orc):
    """The interleaved order's warmup (reading R4), pinned by the timing it is
    built for.  The pages name Megatron's interleaved schedule ("2. 1F1B" §6.1,
    M040 §06) but print neither its order nor its warmup count; the reading
    takes the order whose warmup fills device k with forwards until the first
    gradient can reach it.  Derivation at one tick per op and no latency:
    microbatch 0 enters virtual stage s at tick s, so its forward leaves the
    last of the S = vP virtual stages at tick S; its gradient then walks back
    one virtual stage per tick and reaches virtual stage (v-1)P + k -- device
    k's last chunk, whose backward comes first -- at tick S + (P-1-k).  Device
    k receives its first input at tick k, so it runs S + P - 1 - 2k forwards
    back to back before it (at most the vM it has), then its first backward
    (chunk v-1, microbatch 0) at that tick.  Its ledger peaks there, since each
    later forward is paired with a backward."""
    for P in (1, 2, 3, 4, 5, 8):
        for v in (2, 3, 4):
            for M in (P, 2 * P, 3 * P, 4 * P):
                kind, chunk, mb = orc.order("interleaved", P, M, v)
                r = orc.evaluate("interleaved", P, M, v, 1, 1)
                S = v * P
                for k in range(P):
                    want = min(S + P - 1 - 2 * k, v * M)
                    seq = list(kind[k])
                    first_b = seq.index(1)
                    assert first_b == want, (P, v, M, k)
                    assert r["peak"][k] == want
                    assert (chunk[k][first_b], mb[k][first_b]) == (v - 1, 0)
                    if want < v * M:
                        # no idle tick in the warmup, and the backward at its arrival
                        assert list(r["start"][k][:first_b + 1]) == list(range(k, k + first_b + 1))
                        assert r["start"][k][first_b] == S + P - 1 - k
    # P = 4, v = 2, M = 8: the counts written out
    assert [list(orc.order("interleaved", 4, 8, 2)[0][k]).index(1) for k in range(4)] == [11, 9, 7, 5]


def test_gpipe_comm_invariant(orc):
    # GPipe with every stage equally fast and uniform comm c: the forward wave
    # reaches the last stage after (P-1)(t_f+c) + M t_f, the backward wave needs
    # (P-1)(t_b+c) + M t_b more, so total = (M+P-1)(t_f+t_b) + 2(P-1)c.
    for P in range(1, 7):
        for M in (1, 3, 8):
            for tf, tb, c in ((1, 1, 1), (1, 2, 3), (2, 3, 1)):
                r = orc.evaluate("gpipe", P, M, 1, tf, tb, comm=c, method=2)
                assert r["makespan"] == (M + P - 1) * (tf + tb) + 2 * (P - 1) * c


def _census_by_graph(P, M):
    """Independent enumeration for tiny P, M at unit cost: every combination of
    per-stage orders with each F_i before its B_i, run as a plain dependency
    graph (stage order, F(s-1,i) -> F(s,i), B(s+1,i) -> B(s,i)); a cycle is a
    deadlock, else the makespan is the longest path counted in ops.  Returns
    (valid, deadlocked, min makespan, orders reaching it, min stage-0 peak
    among them)."""
    ops = [(0, i) for i in range(M)] + [(1, i) for i in range(M)]
    stage_orders = [q for q in itertools.permutations(ops)
                    if all(q.index((0, i)) < q.index((1, i)) for i in range(M))]
    valid = dead = 0
    best, nbest, pk0 = None, 0, None
    for combo in itertools.product(stage_orders, repeat=P):
        preds = {}
        for s, q in enumerate(combo):
            for j, (kd, i) in enumerate(q):
                p = [(s, *q[j - 1])] if j else []
                if kd == 0 and s > 0:
                    p.append((s - 1, 0, i))
                if kd == 1 and s < P - 1:
                    p.append((s + 1, 1, i))
                preds[(s, kd, i)] = p
        depth, state = {}, {}

        def longest(node):
            # iterative DFS; returns None on a cycle
            stack = [node]
            while stack:
                x = stack[-1]
                if x in depth:
                    stack.pop()
                    continue
                state[x] = 1
                todo = [y for y in preds[x] if y not in depth]
                for y in todo:
                    if state.get(y) == 1:
                        return None
                if todo:
                    stack.extend(todo)
                    continue
                depth[x] = 1 + max((depth[y] for y in preds[x]), default=0)
                state[x] = 2
                stack.pop()
            return depth[node]

        mk = 0
        for x in preds:
            d = longest(x)
            if d is None:
                mk = None
                break
            mk = max(mk, d)
        if mk is None:
            dead += 1
            continue
        valid += 1
        held, peak0 = 0, 0
        for kd, _ in combo[0]:
            held += 1 if kd == 0 else -1
            peak0 = max(peak0, held)
        if best is None or mk < best:
            best, nbest, pk0 = mk, 0, peak0
        if mk == best:
            nbest += 1
            pk0 = min(pk0, peak0)
    return valid, dead, best, nbest, pk0


def test_bruteforce_optimality(orc):
    # "2. 1F1B" §4.2/§4.3: no valid order beats 2(M+P-1) at unit cost, and no
    # order that is not slower holds fewer than min(P, M) activations on stage 0.
    for P in (1, 2, 3):
        for M in (1, 2, 3):
            b = orc.bruteforce(P, M)
            assert b["min_makespan"] == 2 * (M + P - 1)
            assert b["min_peak0"] == min(P, M)
            for policy in ("gpipe", "1f1b"):
                assert orc.evaluate(policy, P, M, 1, 1, 1)["makespan"] == b["min_makespan"]
            assert orc.evaluate("1f1b", P, M, 1, 1, 1)["peak"][0] == b["min_peak0"]


def test_bruteforce_census(orc):
    """The census of the exhaustive check, cell by cell for P, M <= 3."""
    for P in (1, 2, 3):
        for M in (1, 2, 3):
            b = orc.bruteforce(P, M)
            # A stage runs 2M ops with each F_i before its B_i: (2M)!/2^M orders,
            # independently on each of the P stages.
            assert b["valid"] + b["deadlocked"] == (math.factorial(2 * M) // 2 ** M) ** P
            if P == 1:
                # one stage has no cross-stage edge: nothing deadlocks and every
                # order keeps the stage busy for all 2M ticks
                assert b["deadlocked"] == 0 and b["n_optimal"] == b["valid"]
            if M == 1:
                assert (b["valid"], b["deadlocked"], b["n_optimal"]) == (1, 0, 1)
            if (P, M) != (3, 3):
                # an enumeration of its own (a dependency graph per combination)
                want = _census_by_graph(P, M)
                got = (b["valid"], b["deadlocked"], b["min_makespan"], b["n_optimal"], b["min_peak0"])
                assert got == want, (P, M)
    # P = M = 3: 729,000 combinations, of which 138,294 run, 590,706 deadlock
    # and 210 reach the minimum 10 ticks (an independent enumeration's census).
    b = orc.bruteforce(3, 3)
    assert (b["valid"], b["deadlocked"], b["n_optimal"]) == (138294, 590706, 210)


def test_deadlock_detected_by_both_evaluators(orc):
    # A cyclic order: stage 0 wants B0 before F1, stage 1 wants F1 before F0.
    kind = np.array([[0, 1, 0, 1], [0, 1, 0, 1]], np.int32)
    mb = np.array([[0, 0, 1, 1], [1, 1, 0, 0]], np.int32)
    chunk = np.zeros((2, 4), np.int32)
    for method in (0, 1):
        with pytest.raises(orc.OracleError) as e:
            orc.eval_explicit(2, 2, 1, kind, chunk, mb, 1, 1, method=method)
        assert e.value.code == orc.ERR_DEADLOCK


def test_des_matches_longest_path_random(orc):
    rng = np.random.default_rng(123)
    for _ in range(120):
        policy = rng.choice(["gpipe", "1f1b", "interleaved"])
        P = int(rng.integers(1, 7))
        v = int(rng.integers(2, 4)) if policy == "interleaved" else 1
        M = P * int(rng.integers(1, 4)) if policy == "interleaved" else int(rng.integers(1, 12))
        S = P * v
        tf = rng.integers(0, 9, (S, M))
        tb = rng.integers(0, 9, (S, M))
        cm = rng.integers(0, 5, max(S - 1, 1))
        r = orc.evaluate(policy, P, M, v, tf, tb, comm=cm, method=2)   # raises on mismatch
        # dependency and overlap invariants checked directly here as well
        assert r["makespan"] == r["end"].max()
        for k in range(P):
            assert np.all(r["start"][k, 1:] >= r["end"][k, :-1])


def test_batch_strides_status_and_overflow(orc):
    rng = np.random.default_rng(5)
    P, M, n = 3, 4, 6
    cf = rng.integers(1, 5, (n, P, M)).astype(np.int32)
    cb = rng.integers(1, 5, (n, P, M)).astype(np.int32)
    cf[2, 1, 1] = -1
    cb[4, 0, 0] = 2**31 - 1
    out = orc.eval_batch("1f1b", P, M, 1, cf, cb, (P * M, M, 1), n=n, method=2)
    assert out["status"][2] == orc.ST_NEG_COST
    assert out["status"][4] == orc.ST_OVERFLOW
    for x in (0, 1, 3, 5):
        assert out["status"][x] == orc.ST_OK
        r = orc.evaluate("1f1b", P, M, 1, cf[x], cb[x])
        assert out["makespan"][x] == r["makespan"]
        assert list(out["idle"][x]) == list(r["idle"])
    # instance-minor layout gives the same numbers
    cfT = np.ascontiguousarray(np.transpose(cf, (1, 2, 0)))
    cbT = np.ascontiguousarray(np.transpose(cb, (1, 2, 0)))
    out2 = orc.eval_batch("1f1b", P, M, 1, cfT, cbT, (1, M * n, n), n=n)
    assert np.array_equal(out["makespan"], out2["makespan"])
    assert np.array_equal(out["status"], out2["status"])


def test_splitmix64_published_vector(orc):
    g = read_golden("splitmix64_seed0.txt")
    gamma = 0x9E3779B97F4A7C15
    for n_str, (val,) in g.items():
        n = int(n_str)
        assert orc.splitmix64((gamma * n) % 2**64) == int(val, 16)


def test_binom_and_unranking(orc):
    assert orc.binom(79, 7) == math.comb(79, 7) == 2898753715
    for n in range(0, 30):
        for k in range(0, 8):
            assert orc.binom(n, k) == math.comb(n, k)
    # colex unranking against explicit enumeration: sort all K-subsets of
    # range(N) by their reversed tuple; rank r is the r-th subset.
    for N, K in ((7, 2), (9, 3), (10, 4)):
        subsets = sorted(itertools.combinations(range(N), K), key=lambda s: s[::-1])
        L, P = N + 1, K + 1
        tot = math.comb(N, K)
        for c in range(60):
            u = orc.splitmix64(77 + c)
            first = orc.candidate_split(77, c, L, P)
            x = subsets[u % tot]
            assert list(first) == [0] + [xi + 1 for xi in x] + [L]


def test_search_finds_global_optimum_small(orc):
    rng = np.random.default_rng(9)
    L, P, M = 8, 3, 6
    ltf = rng.integers(5, 15, L).astype(np.int32)
    ltb = (2 * ltf).astype(np.int32)
    lact = rng.integers(1, 4, L).astype(np.int64)
    # brute force over every contiguous split with itertools
    best = None
    for cuts in itertools.combinations(range(1, L), P - 1):
        bounds = [0, *cuts, L]
        tf = [int(ltf[bounds[k]:bounds[k + 1]].sum()) for k in range(P)]
        tb = [int(ltb[bounds[k]:bounds[k + 1]].sum()) for k in range(P)]
        r = orc.evaluate("1f1b", P, M, 1, np.repeat(np.array(tf)[:, None], M, 1),
                         np.repeat(np.array(tb)[:, None], M, 1))
        if best is None or r["makespan"] < best:
            best = r["makespan"]
    res = orc.search(ltf, ltb, lact, P, M, 0, 10**12, 42, 0, 3000)
    assert res["best_makespan"] == best
    assert res["all_makespan"][res["best_idx"]] == best
    assert res["all_makespan"].min() == best
    assert res["first"][0] == 0 and res["first"][-1] == L
    # the cap rejects splits: peak_k * act_k must stay <= cap
    tight = orc.search(ltf, ltb, lact, P, M, 0, 0, 42, 0, 50)
    assert tight["best_idx"] == -1 and (tight["all_makespan"] == -1).all()


def test_exhaustive_search_covers_every_split(orc):
    """Ranks 0 .. C(L-1, P-1)-1 enumerate every contiguous split exactly once,
    rank r being the colex rank sum_i C(x_i, i) of its cut positions (the
    combinatorial number system), and every split is scored as a direct
    1F1B evaluation of its stage sums would score it."""
    rng = np.random.default_rng(19)
    L, P, M, comm = 10, 4, 5, 1
    ltf = rng.integers(3, 12, L).astype(np.int32)
    ltb = rng.integers(5, 25, L).astype(np.int32)
    lact = rng.integers(1, 5, L).astype(np.int64)
    total = math.comb(L - 1, P - 1)
    cap = 30
    res = orc.search_ranks(ltf, ltb, lact, P, M, comm, cap, 0, total)
    seen = set()
    for r in range(total):
        first = [int(v) for v in orc.rank_split(r, L, P)]
        x = [f - 1 for f in first[1:P]]
        assert sum(math.comb(xi, i + 1) for i, xi in enumerate(x)) == r
        seen.add(tuple(first[1:P]))
        tf = [int(ltf[first[k]:first[k + 1]].sum()) for k in range(P)]
        tb = [int(ltb[first[k]:first[k + 1]].sum()) for k in range(P)]
        act = [int(lact[first[k]:first[k + 1]].sum()) for k in range(P)]
        if any(min(P - k, M) * act[k] > cap for k in range(P)):
            assert res["all_makespan"][r] == -1
            continue
        ev = orc.evaluate("1f1b", P, M, 1, np.repeat(np.array(tf)[:, None], M, 1),
                          np.repeat(np.array(tb)[:, None], M, 1), comm)
        assert res["all_makespan"][r] == ev["makespan"]
    assert seen == set(itertools.combinations(range(1, L), P - 1))
    feas = res["all_makespan"] >= 0
    assert feas.any() and not feas.all()
    best = int(res["all_makespan"][feas].min())
    assert res["best_makespan"] == best
    assert res["best_idx"] == int(np.nonzero(res["all_makespan"] == best)[0][0])
    assert list(res["first"]) == [int(v) for v in orc.rank_split(res["best_idx"], L, P)]


def test_interleaved_search_scores_layouts(orc):
    """Each candidate splits the layers into P*v contiguous ranges (virtual
    stage s on device s mod P); its score equals a direct interleaved
    evaluation of the range sums, and it is rejected exactly when a device's
    chunk-weighted held bytes peak above the cap.  With v = 1 the search is
    the 1F1B search."""
    rng = np.random.default_rng(23)
    L, P, v, M, comm = 14, 3, 2, 6, 1
    S = P * v
    ltf = rng.integers(3, 12, L).astype(np.int32)
    ltb = rng.integers(5, 25, L).astype(np.int32)
    lact = rng.integers(1, 5, L).astype(np.int64)
    cap = 40
    res = orc.search_interleaved(ltf, ltb, lact, P, v, M, comm, cap, 99, 0, 120)
    kind, chunk, _ = orc.order("interleaved", P, M, v)
    rejected = 0
    for c in range(120):
        first = [int(x) for x in orc.candidate_split(99, c, L, S)]
        tf = [int(ltf[first[s]:first[s + 1]].sum()) for s in range(S)]
        tb = [int(ltb[first[s]:first[s + 1]].sum()) for s in range(S)]
        act = [int(lact[first[s]:first[s + 1]].sum()) for s in range(S)]
        top = []
        for d in range(P):
            held, hi = 0, 0
            for j in range(kind.shape[1]):
                a = act[chunk[d, j] * P + d]
                held += a if kind[d, j] == 0 else -a
                hi = max(hi, held)
            top.append(hi)
        if max(top) > cap:
            rejected += 1
            assert res["all_makespan"][c] == -1
            continue
        ev = orc.evaluate("interleaved", P, M, v, np.repeat(np.array(tf)[:, None], M, 1),
                          np.repeat(np.array(tb)[:, None], M, 1), comm)
        assert res["all_makespan"][c] == ev["makespan"]
    assert 0 < rejected < 120
    one = orc.search_interleaved(ltf, ltb, lact, P, 1, M, comm, cap, 99, 0, 50)
    base = orc.search(ltf, ltb, lact, P, M, comm, cap, 99, 0, 50)
    assert np.array_equal(one["all_makespan"], base["all_makespan"])


def test_gpipe_fifo_variant(orc):
    """GPipe with first-in-first-out backwards: the same makespan as GPipe's
    last-in-first-out order at costs uniform over microbatches (R1), other op
    times, the same peak M; both evaluators agree on heterogeneous costs."""
    for P, M in ((2, 4), (4, 8), (5, 3), (8, 16)):
        for tf, tb in ((1, 1), (1, 2), (3, 5)):
            fifo = orc.evaluate("gpipe_fifo", P, M, 1, tf, tb)
            lifo = orc.evaluate("gpipe", P, M, 1, tf, tb)
            assert fifo["makespan"] == lifo["makespan"] == (M + P - 1) * (tf + tb)
            assert list(fifo["peak"]) == [M] * P
            # same ticks per position, other microbatches at them: B of
            # microbatch 0 runs first under FIFO and last under LIFO
            assert np.array_equal(fifo["start"], lifo["start"])
            if M > 1:
                assert fifo["mb"][0, M] == 0 and lifo["mb"][0, M] == M - 1
            kind, _, mb = orc.order("gpipe_fifo", P, M)
            assert list(mb[0, M:]) == list(range(M)) and (kind[:, M:] == 1).all()
    rng = np.random.default_rng(29)
    for _ in range(20):
        P, M = int(rng.integers(1, 7)), int(rng.integers(1, 10))
        r = orc.evaluate("gpipe_fifo", P, M, 1, rng.integers(0, 9, (P, M)), rng.integers(0, 9, (P, M)),
                         rng.integers(0, 4, max(P - 1, 1)), method=2)
        assert r["makespan"] >= 0


def test_separate_forward_backward_comm(orc):
    """Forward edges with latency c_f and backward edges with c_b: GPipe at
    uniform costs ends at (M+P-1)(t_f+t_b) + (P-1)(c_f+c_b) (the forward chain
    crosses P-1 forward edges and the gradient chain P-1 backward edges; the
    case c_f = c_b is the invariant above); c_b = c_f everywhere equals a
    single comm; both evaluators agree on heterogeneous inputs."""
    for P, M in ((2, 3), (4, 8), (6, 5)):
        for cf_, cb_ in ((1, 4), (3, 0), (2, 2)):
            r = orc.evaluate("gpipe", P, M, 1, 2, 3, cf_, comm_b=cb_)
            assert r["makespan"] == (M + P - 1) * 5 + (P - 1) * (cf_ + cb_)
    rng = np.random.default_rng(31)
    for _ in range(30):
        P, M = int(rng.integers(1, 6)), int(rng.integers(1, 9))
        pol = ["gpipe", "1f1b", "gpipe_fifo"][int(rng.integers(0, 3))]
        tf, tb = rng.integers(0, 9, (P, M)), rng.integers(0, 9, (P, M))
        c = rng.integers(0, 5, max(P - 1, 1))
        a = orc.evaluate(pol, P, M, 1, tf, tb, c, comm_b=c, method=2)
        b = orc.evaluate(pol, P, M, 1, tf, tb, c, method=2)
        assert np.array_equal(a["start"], b["start"])
        orc.evaluate(pol, P, M, 1, tf, tb, c, comm_b=rng.integers(0, 5, max(P - 1, 1)), method=2)


MUTANTS = {
    1: "forward edges carry no comm",
    2: "1F1B warmup off by one",
    3: "GPipe backward FIFO",
    4: "B ignores downstream gradient",
    5: "ledger sign flipped",
    6: "bubble over ideal time",
    7: "splitmix64 shift mistyped",
    8: "unranking off by one",
    9: "ZB runs a pending W before a ready F/B",
    10: "ZB2P keeps 1F1B's warmup",
    11: "ZB admits an F at the activation limit",
    12: "backward edges take the forward latency",
    13: "interleaved warmup one forward too long",
    14: "DualPipe runs a ready forward before a ready backward",
    15: "DualPipe route B crosses a boundary on route A's link",
    16: "search rejects a layout exactly at the byte cap",
    17: "search breaks a makespan tie toward the later candidate",
    18: "interleaved search weighs every op by the device's first chunk",
}


def _pin_suite(orc, lib):
    """Run a compact version of the pins above against a given library;
    returns the list of pins that fail."""
    failed = []

    def check(name, fn):
        try:
            ok = fn()
        except Exception:
            ok = False
        if not ok:
            failed.append(name)

    def tables():
        for policy, fx in (("gpipe", "m040_gpipe_2x4.txt"), ("1f1b", "m040_1f1b_2x4.txt")):
            g = read_golden(fx)
            r = orc.evaluate(policy, 2, 4, 1, 1, 1, lib=lib)
            if _table_from_oracle(r, 2) != [g["stage0"], g["stage1"]]:
                return False
            if r["peak"][0] != int(g["peak_stage0"][0]):
                return False
        return True

    def closed():
        for policy in ("gpipe", "1f1b"):
            r = orc.evaluate(policy, 4, 8, 1, 1, 1, lib=lib)
            if r["makespan"] != 22 or Fraction(*r["bub"]) != Fraction(3, 11):
                return False
        return True

    def comm():
        r = orc.evaluate("gpipe", 4, 3, 1, 1, 2, comm=3, lib=lib)
        return r["makespan"] == 6 * 3 + 2 * 3 * 3

    def phases():
        kind, _, _ = orc.order("1f1b", 4, 8, lib=lib)
        return [list(kind[k]).index(1) for k in range(4)] == [4, 3, 2, 1]

    def sm():
        return orc.splitmix64(0, lib=lib) == 0xE220A8397B1DCDAF

    def unrank():
        subsets = sorted(itertools.combinations(range(9), 3), key=lambda s: s[::-1])
        for c in range(40):
            first = orc.candidate_split(5, c, 10, 4, lib=lib)
            x = subsets[orc.splitmix64(5 + c, lib=lib) % math.comb(9, 3)]
            if list(first) != [0] + [xi + 1 for xi in x] + [10]:
                return False
        return True

    def zb():
        from test_oracle_zb import zb_tick_sim
        for policy, fx in (("zb1p", "zb1p_p2m2_unit.txt"), ("zb2p", "zb2p_p2m2_unit.txt")):
            g = read_golden(fx)
            r = orc.zb_evaluate(policy, 2, 2, 1, 1, 1, lib=lib)
            if r["makespan"] != int(g["makespan"][0]) or r["bub"] != tuple(int(x) for x in g["bubble"]):
                return False
        rng = np.random.default_rng(21)
        for policy in ("zb1p", "zb2p"):
            for P, M in ((2, 4), (3, 6), (4, 9)):
                tf = rng.integers(1, 4, size=(P, M))
                tb = rng.integers(1, 4, size=(P, M))
                tw = rng.integers(3, 9, size=(P, M))
                cm = rng.integers(0, 3, size=P - 1)
                r = orc.zb_evaluate(policy, P, M, tf, tb, tw, cm, lib=lib)
                S, _, _ = zb_tick_sim(policy, P, M, tf, tb, tw, cm)
                if not np.array_equal(r["start"], S):
                    return False
        return True

    check("tables", tables)
    check("closed", closed)
    check("comm", comm)
    check("phases", phases)
    check("splitmix", sm)
    check("unrank", unrank)
    check("zb", zb)

    def comm_fb():
        r = orc.evaluate("gpipe", 4, 8, 1, 2, 3, 1, lib=lib, comm_b=4)
        return r["makespan"] == 11 * 5 + 3 * 5

    check("comm_fb", comm_fb)

    def ilv_warmup():
        P, M, v = 4, 8, 2
        kind, chunk, _ = orc.order("interleaved", P, M, v, lib=lib)
        r = orc.evaluate("interleaved", P, M, v, 1, 1, lib=lib)
        want = [min(v * P + P - 1 - 2 * k, v * M) for k in range(P)]
        return ([list(kind[k]).index(1) for k in range(P)] == want
                and list(r["peak"]) == want)

    check("ilv_warmup", ilv_warmup)

    def dualpipe():
        from test_oracle_dualpipe import dp_tick_sim
        rng = np.random.default_rng(8)
        for P, MA, MB in ((4, 5, 4), (3, 2, 4), (6, 7, 7)):
            M = MA + MB
            tf = rng.integers(1, 5, size=(P, M))
            tb = rng.integers(1, 5, size=(P, M))
            cm = rng.integers(0, 4, size=P - 1)
            r = orc.dp_evaluate(P, MA, MB, tf, tb, cm, lib=lib)
            if not np.array_equal(r["start"], dp_tick_sim(P, MA, MB, tf, tb, cm)[0]):
                return False
        r = orc.dp_evaluate(8, 16, 16, 1, 2, lib=lib)
        return list(r["idle"]) == [3 * 5] * 8

    check("dualpipe", dualpipe)

    def search_cap():
        # reading R11: stage k holds min(P-k, M) microbatches of its layers'
        # bytes at its peak; a layout is rejected only when that exceeds the
        # cap (a layout exactly at the cap is kept)
        P, L, M = 3, 6, 4
        ltf = np.ones(L, np.int32)
        ltb = np.full(L, 2, np.int32)
        lact = np.array([5, 1, 3, 2, 4, 6], np.int64)
        C = math.comb(L - 1, P - 1)
        need = []
        for r in range(C):
            f = list(orc.rank_split(r, L, P, lib=lib))
            need.append(max(min(P - k, M) * int(lact[f[k]:f[k + 1]].sum()) for k in range(P)))
        cap = sorted(set(need))[len(set(need)) // 2]
        res = orc.search_ranks(ltf, ltb, lact, P, M, 0, cap, 0, C, lib=lib)
        return all((int(res["all_makespan"][r]) == -1) == (need[r] > cap) for r in range(C))

    def search_tie():
        # with one microbatch every split runs the same chain of all forwards
        # then all backwards: every makespan ties and the lowest rank wins
        L, P = 6, 3
        C = math.comb(L - 1, P - 1)
        res = orc.search_ranks(np.arange(1, L + 1, dtype=np.int32), np.full(L, 3, np.int32), np.ones(L, np.int64),
                               P, 1, 0, 10**12, 0, C, lib=lib)
        mks = set(int(x) for x in res["all_makespan"])
        return mks == {int(np.arange(1, L + 1).sum()) + 3 * L} and res["best_idx"] == 0

    def ilv_ledger():
        # reading R22: each device's held bytes run over its interleaved order,
        # + the bytes of the op's range at F, - at B; reject above the cap
        P, v, M, L = 2, 2, 4, 11
        S = P * v
        rng = np.random.default_rng(31)
        ltf = rng.integers(1, 9, L).astype(np.int32)
        ltb = rng.integers(1, 9, L).astype(np.int32)
        lact = rng.integers(1, 50, L).astype(np.int64)
        kind, chunk, _ = orc.order("interleaved", P, M, v, lib=lib)
        tops = []
        for c in range(60):
            f = list(orc.candidate_split(9, c, L, S, lib=lib))
            act = [int(lact[f[q]:f[q + 1]].sum()) for q in range(S)]
            top = 0
            for d in range(P):
                held = 0
                for j in range(2 * M * v):
                    held += (1 if kind[d][j] == 0 else -1) * act[chunk[d][j] * P + d]
                    top = max(top, held)
            tops.append(top)
        cap = int(np.median(tops))
        res = orc.search_interleaved(ltf, ltb, lact, P, v, M, 0, cap, 9, 0, 60, lib=lib)
        return all((int(res["all_makespan"][c]) == -1) == (tops[c] > cap) for c in range(60))

    check("search_cap", search_cap)
    check("search_tie", search_tie)
    check("ilv_ledger", ilv_ledger)
    return failed


def test_pins_pass_on_oracle(orc):
    assert _pin_suite(orc, orc.load()) == []


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(orc, mutant):
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, f"liborc_m{mutant}.so")
        orc.build(path, defines=(f"ORC_MUTANT={mutant}",))
        lib = orc.load(path)
        failed = _pin_suite(orc, lib)
    assert failed, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"


def test_1f1b_makespan_lower_bound(orc):
    """The bound the GPU searches prune with, checked on the oracle: for 1F1B
    with stage costs f_k, b_k >= 0 and latency c on every boundary, stage k
    runs 2M ops one at a time between microbatch 0's forward arriving (after
    sum_{j<k} f_j + k c) and the last backward leaving (sum_{j<k} b_j + k c
    before the end), so makespan >= max_k [sum_{j<k} (f_j + b_j) + 2 k c +
    M (f_k + b_k)].  It is exact for a single stage; a bound one microbatch
    too large (M + 1 in place of M) fails on some instance, so the check is not
    vacuous."""
    rng = np.random.default_rng(77)
    too_big_fails = False
    for _ in range(400):
        P = int(rng.integers(1, 9))
        M = int(rng.integers(1, 20))
        c = int(rng.integers(0, 4))
        f = rng.integers(0, 30, P)
        b = rng.integers(0, 60, P)
        r = orc.evaluate("1f1b", P, M, 1, f[:, None], b[:, None], comm=c)
        pre, lb = 0, 0
        for k in range(P):
            lb = max(lb, pre + M * (int(f[k]) + int(b[k])))
            pre += int(f[k]) + int(b[k]) + 2 * c
        assert r["makespan"] >= lb
        if P == 1:
            assert r["makespan"] == lb
        pre, lb1 = 0, 0
        for k in range(P):
            lb1 = max(lb1, pre + (M + 1) * (int(f[k]) + int(b[k])))
            pre += int(f[k]) + int(b[k]) + 2 * c
        too_big_fails |= r["makespan"] < lb1
    assert too_big_fails


def test_interleaved_makespan_lower_bound(orc):
    """The bound the interleaved search prunes with, checked on the oracle:
    with M a multiple of P, device d's first op is microbatch 0's forward of
    its chunk 0 (virtual stage d) and its last op the backward of chunk 0 for
    microbatch M - 1, and it runs all 2 M v of its ops one at a time, so
    makespan >= max_d [sum_{s<d} (f_s + b_s) + 2 d c + M sum_chunks (f + b)]
    (virtual stage s = chunk * P + d).  A bound one microbatch too large fails
    somewhere."""
    rng = np.random.default_rng(78)
    too_big_fails = False
    for _ in range(300):
        P = int(rng.integers(1, 6))
        v = int(rng.integers(2, 4))
        M = P * int(rng.integers(1, 4))
        c = int(rng.integers(0, 4))
        f = rng.integers(0, 30, P * v)
        b = rng.integers(0, 60, P * v)
        r = orc.evaluate("interleaved", P, M, v, f[:, None], b[:, None], comm=c)
        for extra, check in ((0, True), (1, False)):
            lb, pre = 0, 0
            for d in range(P):
                busy = sum(int(f[ch * P + d]) + int(b[ch * P + d]) for ch in range(v))
                lb = max(lb, pre + 2 * d * c + (M + extra) * busy)
                pre += int(f[d]) + int(b[d])
            if check:
                assert r["makespan"] >= lb
            else:
                too_big_fails |= r["makespan"] < lb
    assert too_big_fails


def test_interleaved_ledger_peak_from_dominant_counts(orc):
    """The identity the interleaved search's byte cap relies on, checked on the
    oracle's orders: for non-negative chunk bytes, the peak of the ledger (+ a
    chunk's bytes at its F, - at its B, [1F1B] §4.1 weighted) over a device's
    order equals the largest dot product of the bytes with the held-count
    vectors of the order that no other vector dominates; with a negative byte
    count it may not, which is why the search walks the order then."""
    rng = np.random.default_rng(79)
    differs = False
    for P, M, v in ((2, 4, 2), (3, 6, 3), (4, 8, 2), (8, 16, 4), (5, 10, 2)):
        kind, chunk, mb = orc.order("interleaved", P, M, v)
        for d in range(P):
            h = np.zeros(v, np.int64)
            path = [h.copy()]
            for j in range(kind.shape[1]):
                h[chunk[d, j]] += 1 if kind[d, j] == 0 else -1
                path.append(h.copy())
            vecs = np.unique(np.array(path), axis=0)
            dom = np.array([x for x in vecs if not any((y >= x).all() and (y != x).any() for y in vecs)])
            for _ in range(40):
                act = rng.integers(0, 1000, v)
                walk = max(int(p @ act) for p in path)
                assert walk == max(int(x @ act) for x in dom)
                neg = rng.integers(-1000, 1000, v)
                differs |= max(int(p @ neg) for p in path) != max(int(x @ neg) for x in dom)
    assert differs
