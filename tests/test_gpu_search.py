"""GPU partition search against the oracle's candidate scorer (bit-exact
makespans, identical argmin with ties to the lower candidate index)."""
import math
import os

import numpy as np
import pytest
import torch

import pipeline_schedule_simulation_gb300.workloads as W
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from pipeline_schedule_simulation_gb300 import binding
    return binding


def _gpu_search(B, p, begin, n, all_mk=True):
    out = B.partition_search(to_dev(p.layer_tf), to_dev(p.layer_tb), to_dev(p.layer_act), p.P, p.M,
                             p.comm, p.cap, p.seed, begin, n, all_makespan=all_mk)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("L,P,M,comm,cap", [(8, 3, 6, 0, 10**12), (20, 5, 10, 2, 9), (12, 1, 4, 0, 10**9),
                                            (30, 8, 16, 1, 40), (40, 16, 20, 0, 10**12)])
def test_small_exact(orc, B, L, P, M, comm, cap):
    rng = np.random.default_rng(L + P)
    p = W.SearchProblem(rng.integers(1, 20, L).astype(np.int32), rng.integers(1, 40, L).astype(np.int32),
                        rng.integers(1, 4, L).astype(np.int64), P, M, comm, cap, 1234 + L, 0)
    n = 3000
    g = _gpu_search(B, p, 0, n)
    r = orc.search(p.layer_tf, p.layer_tb, p.layer_act, P, M, comm, cap, p.seed, 0, n, nthreads=8)
    assert np.array_equal(g["all_makespan"], r["all_makespan"])
    assert int(g["best_idx"][0]) == r["best_idx"]
    assert int(g["best_makespan"][0]) == r["best_makespan"]
    if P > 1 and r["best_idx"] >= 0:
        assert list(g["best_cuts"]) == list(r["first"][1:P])


def test_nothing_feasible(B):
    p = W.SearchProblem(np.full(10, 5, np.int32), np.full(10, 9, np.int32), np.full(10, 100, np.int64),
                        4, 8, 0, 10, 7, 0)
    g = _gpu_search(B, p, 0, 500)
    assert g["best_idx"][0] == -1 and g["best_makespan"][0] == -1
    assert (g["best_cuts"] == -1).all() and (g["all_makespan"] == -1).all()


def test_layer_split_full(orc, B):
    """1,048,576 candidates of the 80-layer model at P=8, M=128: every
    candidate's makespan (or rejection) equals the oracle's, and so do the
    argmin (lowest index of the minimum), its makespan and its stage split."""
    p = W.layer_split()
    g = _gpu_search(B, p, 0, p.n_cand)
    r = orc.search(p.layer_tf, p.layer_tb, p.layer_act, p.P, p.M, p.comm, p.cap, p.seed, 0, p.n_cand,
                   nthreads=os.cpu_count() or 8)
    mk = g["all_makespan"]
    assert np.array_equal(mk, r["all_makespan"])
    assert (mk >= 0).any()
    assert int(g["best_idx"][0]) == r["best_idx"]
    assert int(g["best_makespan"][0]) == r["best_makespan"]
    assert list(g["best_cuts"]) == list(r["first"][1:p.P])


def test_split_ranges_reduce_to_whole(B):
    from pipeline_schedule_simulation_gb300.sharding import best_of
    p = W.layer_split(n_cand=1 << 16)
    whole = _gpu_search(B, p, 0, p.n_cand, all_mk=False)
    parts = []
    for lo, hi in ((0, 30000), (30000, 1 << 16)):
        g = _gpu_search(B, p, lo, hi - lo, all_mk=False)
        parts.append((int(g["best_makespan"][0]), int(g["best_idx"][0])))
    assert best_of(parts) == (int(whole["best_makespan"][0]), int(whole["best_idx"][0]))


@pytest.mark.parametrize("L,P,M,comm,cap", [(10, 4, 5, 1, 30), (20, 5, 10, 2, 10**12), (12, 1, 4, 0, 10**9),
                                            (18, 8, 16, 1, 60), (20, 16, 20, 0, 10**12), (30, 3, 7, 3, 10**12)])
def test_exhaustive_small_exact(orc, B, L, P, M, comm, cap):
    """Every split of small problems, ranks split over two calls: makespans
    bit-exact, best rank and cuts as the oracle's exhaustive search."""
    import math
    rng = np.random.default_rng(L * 7 + P)
    ltf = rng.integers(1, 20, L).astype(np.int32)
    ltb = rng.integers(1, 40, L).astype(np.int32)
    lact = rng.integers(1, 4, L).astype(np.int64)
    total = math.comb(L - 1, P - 1)
    half = total // 2
    got, parts = [], []
    for lo, hi in ((0, half), (half, total)):
        g = B.partition_search_ranks(to_dev(ltf), to_dev(ltb), to_dev(lact), P, M, comm, cap, lo, hi - lo,
                                     all_makespan=True)
        torch.cuda.synchronize()
        got.append(g["all_makespan"].cpu().numpy())
        parts.append((int(g["best_makespan"].item()), int(g["best_idx"].item())))
    allmk = np.concatenate(got)
    r = orc.search_ranks(ltf, ltb, lact, P, M, comm, cap, 0, total, nthreads=8)
    assert np.array_equal(allmk, r["all_makespan"])
    from pipeline_schedule_simulation_gb300.sharding import best_of
    feas = [p for p in parts if p[1] >= 0]
    if r["best_idx"] >= 0:
        assert best_of(feas) == (r["best_makespan"], r["best_idx"])
    whole = B.partition_search_ranks(to_dev(ltf), to_dev(ltb), to_dev(lact), P, M, comm, cap, 0, total)
    torch.cuda.synchronize()
    assert int(whole["best_idx"].item()) == r["best_idx"]
    assert int(whole["best_makespan"].item()) == r["best_makespan"]
    if P > 1 and r["best_idx"] >= 0:
        assert list(whole["best_cuts"].cpu().numpy()) == list(r["first"][1:P])


def test_exhaustive_layer_split_full(orc, B):
    """All 2,898,753,715 splits of the 80-layer model into 8 stages at M=128:
    the winner and 20 sampled rank windows re-scored by the oracle; two halves
    reduce to the whole; no split beats the seeded search's best."""
    import math
    p = W.layer_split()
    total = math.comb(len(p.layer_tf) - 1, p.P - 1)
    assert total == 2_898_753_715
    args = (to_dev(p.layer_tf), to_dev(p.layer_tb), to_dev(p.layer_act), p.P, p.M, p.comm, p.cap)
    whole = B.partition_search_ranks(*args, 0, total)
    torch.cuda.synchronize()
    best, mk = int(whole["best_idx"].item()), int(whole["best_makespan"].item())
    assert best >= 0
    r = orc.search_ranks(p.layer_tf, p.layer_tb, p.layer_act, p.P, p.M, p.comm, p.cap, best, best + 1)
    assert r["best_makespan"] == mk
    assert list(whole["best_cuts"].cpu().numpy()) == list(r["first"][1:p.P])
    seeded = B.partition_search(*args, p.seed, 0, p.n_cand)
    torch.cuda.synchronize()
    assert mk <= int(seeded["best_makespan"].item())
    rng = np.random.default_rng(77)
    for lo in rng.integers(0, total - 16, 20):
        g = B.partition_search_ranks(*args, int(lo), 16, all_makespan=True)
        torch.cuda.synchronize()
        rs = orc.search_ranks(p.layer_tf, p.layer_tb, p.layer_act, p.P, p.M, p.comm, p.cap, int(lo), int(lo) + 16)
        assert np.array_equal(g["all_makespan"].cpu().numpy(), rs["all_makespan"])
    half = total // 2
    parts = []
    for lo, hi in ((0, half), (half, total)):
        g = B.partition_search_ranks(*args, lo, hi - lo)
        torch.cuda.synchronize()
        parts.append((int(g["best_makespan"].item()), int(g["best_idx"].item())))
    from pipeline_schedule_simulation_gb300.sharding import best_of
    assert best_of([q for q in parts if q[1] >= 0]) == (mk, best)


@pytest.mark.parametrize("L,P,v,M,comm,cap", [(14, 3, 2, 6, 1, 40), (20, 4, 2, 8, 2, 10**12), (24, 2, 4, 4, 0, 60),
                                              (40, 8, 2, 16, 1, 10**12), (70, 16, 3, 16, 2, 10**12)])
def test_interleaved_search_exact(orc, B, L, P, v, M, comm, cap):
    """Seeded interleaved layouts: every makespan (rejected, scored) and the
    winner equal the oracle's."""
    rng = np.random.default_rng(L + 3 * P + v)
    ltf = rng.integers(1, 20, L).astype(np.int32)
    ltb = rng.integers(1, 40, L).astype(np.int32)
    lact = rng.integers(1, 4, L).astype(np.int64)
    n = 1500
    g = B.partition_search_interleaved(to_dev(ltf), to_dev(ltb), to_dev(lact), P, v, M, comm, cap, 4321, 0, n,
                                       all_makespan=True)
    torch.cuda.synchronize()
    r = orc.search_interleaved(ltf, ltb, lact, P, v, M, comm, cap, 4321, 0, n, nthreads=8)
    assert np.array_equal(g["all_makespan"].cpu().numpy(), r["all_makespan"])
    assert int(g["best_idx"].item()) == r["best_idx"]
    assert int(g["best_makespan"].item()) == r["best_makespan"]
    if r["best_idx"] >= 0:
        assert list(g["best_cuts"].cpu().numpy()) == list(r["first"][1:P * v])


def test_interleaved_search_chunks_and_ranges(orc, B):
    """More candidates than one scratch chunk (262,144): sampled makespans
    against the oracle, and two ranges reduce to the whole."""
    rng = np.random.default_rng(5)
    L, P, v, M = 30, 2, 2, 4
    ltf = rng.integers(1, 30, L).astype(np.int32)
    ltb = rng.integers(1, 60, L).astype(np.int32)
    lact = rng.integers(1, 4, L).astype(np.int64)
    n = 600_000
    cap = 100
    args = (to_dev(ltf), to_dev(ltb), to_dev(lact), P, v, M, 1, cap, 77)
    whole = B.partition_search_interleaved(*args, 0, n, all_makespan=True)
    torch.cuda.synchronize()
    mk = whole["all_makespan"].cpu().numpy()
    for lo in (0, 262_140, 524_280, n - 40):
        r = orc.search_interleaved(ltf, ltb, lact, P, v, M, 1, cap, 77, lo, lo + 40)
        assert np.array_equal(mk[lo:lo + 40], r["all_makespan"])
    feas = mk >= 0
    assert feas.any() and not feas.all()
    best = int(whole["best_idx"].item())
    assert mk[best] == mk[feas].min() == int(whole["best_makespan"].item())
    assert best == int(np.nonzero(mk == mk[feas].min())[0][0])
    parts = []
    for lo, hi in ((0, 250_000), (250_000, n)):
        g = B.partition_search_interleaved(*args, lo, hi - lo)
        torch.cuda.synchronize()
        parts.append((int(g["best_makespan"].item()), int(g["best_idx"].item())))
    from pipeline_schedule_simulation_gb300.sharding import best_of
    assert best_of(parts) == (int(whole["best_makespan"].item()), best)


def test_interleaved_search_layer_split(orc, B):
    """The 80-layer model as 16 virtual stages (P=8, v=2, M=128), 65,536
    layouts: the winner and 40 sampled layouts re-scored by the oracle."""
    p = W.layer_split()
    args = (to_dev(p.layer_tf), to_dev(p.layer_tb), to_dev(p.layer_act), p.P, 2, p.M, p.comm, p.cap, p.seed)
    g = B.partition_search_interleaved(*args, 0, 1 << 16, all_makespan=True)
    torch.cuda.synchronize()
    mk = g["all_makespan"].cpu().numpy()
    best = int(g["best_idx"].item())
    assert best >= 0 and mk[best] == mk[mk >= 0].min()
    r = orc.search_interleaved(p.layer_tf, p.layer_tb, p.layer_act, p.P, 2, p.M, p.comm, p.cap, p.seed,
                               best, best + 1)
    assert r["best_makespan"] == int(g["best_makespan"].item())
    assert list(g["best_cuts"].cpu().numpy()) == list(r["first"][1:16])
    for lo in np.random.default_rng(3).choice((1 << 16) - 8, 5, replace=False):
        rs = orc.search_interleaved(p.layer_tf, p.layer_tb, p.layer_act, p.P, 2, p.M, p.comm, p.cap, p.seed,
                                    int(lo), int(lo) + 8, nthreads=8)
        assert np.array_equal(mk[lo:lo + 8], rs["all_makespan"])


@pytest.mark.parametrize("comm", [0, 3])
def test_pruned_search_equals_full_scoring(B, comm):
    """Without all_makespan the searches skip candidates whose 1F1B lower
    bound exceeds the best makespan found so far; with it they score every
    candidate.  Both must return the same winner: the seeded 80-layer search
    (1,048,576 candidates) and an exhaustive window of 2^26 splits."""
    p = W.layer_split()
    d = [to_dev(x) for x in (p.layer_tf, p.layer_tb, p.layer_act)]
    keys = ("best_idx", "best_makespan", "best_cuts")
    full = B.partition_search(*d, p.P, p.M, comm, p.cap, p.seed, 0, p.n_cand, all_makespan=True)
    pruned = B.partition_search(*d, p.P, p.M, comm, p.cap, p.seed, 0, p.n_cand)
    n = 1 << 26
    e_full = B.partition_search_ranks(*d, p.P, p.M, comm, p.cap, 123456, n, all_makespan=True)
    e_pruned = B.partition_search_ranks(*d, p.P, p.M, comm, p.cap, 123456, n)
    torch.cuda.synchronize()
    for x, y in ((full, pruned), (e_full, e_pruned)):
        for k in keys:
            assert torch.equal(x[k].cpu(), y[k].cpu()), k
    mk = full["all_makespan"].cpu().numpy()
    assert int(full["best_makespan"].item()) == mk[mk >= 0].min()
    mk = e_full["all_makespan"].cpu().numpy()
    assert int(e_full["best_makespan"].item()) == mk[mk >= 0].min()


def test_interleaved_search_negative_bytes(orc, B):
    """Layouts whose ranges include negative activation bytes take the full
    ledger walk instead of the per-plan table of dominant held counts; mixed
    signs and a binding cap, every makespan against the oracle."""
    rng = np.random.default_rng(11)
    L, P, v, M, cap = 24, 4, 2, 8, 60
    ltf = rng.integers(1, 20, L).astype(np.int32)
    ltb = rng.integers(1, 40, L).astype(np.int32)
    lact = rng.integers(-3, 5, L).astype(np.int64)
    n = 3000
    g = B.partition_search_interleaved(to_dev(ltf), to_dev(ltb), to_dev(lact), P, v, M, 1, cap, 99, 0, n,
                                       all_makespan=True)
    torch.cuda.synchronize()
    r = orc.search_interleaved(ltf, ltb, lact, P, v, M, 1, cap, 99, 0, n, nthreads=8)
    mk = g["all_makespan"].cpu().numpy()
    assert np.array_equal(mk, r["all_makespan"])
    assert (mk == -1).any() and (mk >= 0).any()
    assert int(g["best_idx"].item()) == r["best_idx"]


@pytest.mark.parametrize("comm", [0, 3])
def test_pruned_interleaved_search_equals_full_scoring(B, comm):
    """Without all_makespan the interleaved search skips, from its second
    chunk of 262,144 candidates on, layouts whose interleaved makespan bound
    exceeds the best so far; with it every layout within the cap is scored.
    The same winner either way (1,048,576 layouts of the 80-layer model)."""
    p = W.layer_split()
    d = [to_dev(x) for x in (p.layer_tf, p.layer_tb, p.layer_act)]
    args = (*d, p.P, 2, p.M, comm, p.cap, p.seed, 0, 1 << 20)
    full = B.partition_search_interleaved(*args, all_makespan=True)
    pruned = B.partition_search_interleaved(*args)
    torch.cuda.synchronize()
    for k in ("best_idx", "best_makespan", "best_cuts"):
        assert torch.equal(full[k].cpu(), pruned[k].cpu()), k
    mk = full["all_makespan"].cpu().numpy()
    assert int(full["best_makespan"].item()) == mk[mk >= 0].min()


def test_cap_boundary_and_ties(orc, B):
    """Boundaries the random problems rarely hit: a cap exactly equal to some
    layouts' peak bytes (kept, reading R11; one byte less rejects them), and a
    problem where every split ties (one microbatch: the same chain of all
    forwards then all backwards), where the lowest rank must win; the same
    for the interleaved search with the cap at the median layout's bytes."""
    L, P, M = 12, 4, 6
    rng = np.random.default_rng(41)
    ltf = rng.integers(1, 9, L).astype(np.int32)
    ltb = rng.integers(1, 9, L).astype(np.int32)
    lact = rng.integers(1, 20, L).astype(np.int64)
    C = math.comb(L - 1, P - 1)
    need = []
    for r in range(C):
        f = list(orc.rank_split(r, L, P))
        need.append(max(min(P - k, M) * int(lact[f[k]:f[k + 1]].sum()) for k in range(P)))
    dev = [to_dev(x) for x in (ltf, ltb, lact)]
    for cap in (sorted(need)[C // 2], sorted(need)[C // 2] - 1):
        g = B.partition_search_ranks(*dev, P, M, 1, cap, 0, C, all_makespan=True)
        r = orc.search_ranks(ltf, ltb, lact, P, M, 1, cap, 0, C, nthreads=8)
        am = g["all_makespan"].cpu().numpy()
        assert np.array_equal(am, r["all_makespan"])
        assert np.array_equal(am == -1, np.array(need) > cap)
        assert int(g["best_idx"].item()) == r["best_idx"]
    g = B.partition_search_ranks(*dev, P, 1, 0, 10**15, 0, C, all_makespan=True)
    am = g["all_makespan"].cpu().numpy()
    assert len(set(am.tolist())) == 1 and int(g["best_idx"].item()) == 0
    g = B.partition_search(*dev, P, 1, 0, 10**15, 5, 0, 4000, all_makespan=True)
    assert int(g["best_idx"].item()) == 0
    # interleaved (P divides M): cap at the median of the layouts' own byte peaks
    v, S, M = 2, P * 2, 8
    r0 = orc.search_interleaved(ltf, ltb, lact, P, v, M, 1, 10**15, 3, 0, 400, nthreads=8)
    kind, chunk, _ = orc.order("interleaved", P, M, v)
    tops = []
    for c in range(400):
        f = list(orc.candidate_split(3, c, L, S))
        act = [int(lact[f[q]:f[q + 1]].sum()) for q in range(S)]
        top = 0
        for d in range(P):
            held = 0
            for j in range(2 * M * v):
                held += (1 if kind[d][j] == 0 else -1) * act[chunk[d][j] * P + d]
                top = max(top, held)
        tops.append(top)
    assert (r0["all_makespan"] >= 0).all()
    cap = int(np.median(tops))
    g = B.partition_search_interleaved(*dev, P, v, M, 1, cap, 3, 0, 400, all_makespan=True)
    am = g["all_makespan"].cpu().numpy()
    r = orc.search_interleaved(ltf, ltb, lact, P, v, M, 1, cap, 3, 0, 400, nthreads=8)
    assert np.array_equal(am, r["all_makespan"])
    assert np.array_equal(am == -1, np.array(tops) > cap)
