"""Timeline export (host formatting of op times), checked on op times the
oracle computes; no GPU needed."""
import csv
import json

import numpy as np

from pipeline_schedule_simulation_gb300 import timeline as T


def _packed(kind, chunk, mb):
    return (np.asarray(kind, np.int64) << 31) | (np.asarray(chunk, np.int64) << 24) | np.asarray(mb, np.int64)


def test_records_and_trace_from_plan_order(orc, tmp_path):
    r = orc.evaluate("interleaved", 2, 4, 2, 1, 2, 1)
    ops = _packed(r["kind"], r["chunk"], r["mb"])
    recs = T.records(r["start"], r["end"], ops)
    assert len(recs) == 2 * 16
    for rec in recs:
        assert rec["end"] - rec["start"] == (1 if rec["kind"] == "F" else 2)
    # per device, records are in time order and do not overlap
    for k in range(2):
        dev = [x for x in recs if x["device"] == k]
        assert all(a["end"] <= b["start"] for a, b in zip(dev, dev[1:]))
    tr = T.chrome_trace(recs, us_per_tick=10)
    ev = [e for e in tr["traceEvents"] if e["ph"] == "X"]
    assert len(ev) == 32 and max(e["ts"] + e["dur"] for e in ev) == 10 * r["makespan"]
    assert {e["cat"] for e in ev} == {"F", "B"}
    p = tmp_path / "t.json"
    T.write_chrome_trace(p, recs)
    assert json.loads(p.read_text())["traceEvents"][0]["ph"] == "M"
    c = tmp_path / "t.csv"
    T.write_csv(c, recs)
    rows = list(csv.DictReader(open(c)))
    assert len(rows) == 32 and rows[0].keys() == {"device", "kind", "chunk", "mb", "start", "end", "phase"}


def test_records_zero_bubble(orc):
    r = orc.zb_evaluate("zb1p", 2, 2, 1, 1, 1)
    recs = T.records(r["start"], r["end"], zb=True)
    assert len(recs) == 12
    assert [x["kind"] + str(x["mb"]) for x in recs if x["device"] == 0] == ["F0", "F1", "B0", "W0", "B1", "W1"]


def test_records_dualpipe(orc, tmp_path):
    """DualPipe op times by (block, kind, microbatch) become per-device records:
    route A's block s on device s, route B's on device P-1-s; on every device
    the records are in time order without overlap, and each device holds both
    routes' ops."""
    rng = np.random.default_rng(3)
    P, MA, MB = 4, 5, 4
    r = orc.dp_evaluate(P, MA, MB, rng.integers(1, 5, (P, MA + MB)), rng.integers(1, 5, (P, MA + MB)),
                        rng.integers(0, 3, P - 1))
    recs = T.records(r["start"], r["end"], dualpipe_m_a=MA)
    assert len(recs) == 2 * P * (MA + MB)
    for k in range(P):
        dev = [x for x in recs if x["device"] == k]
        assert len(dev) == 2 * (MA + MB)
        assert {x["route"] for x in dev} == {"A", "B"}
        assert all(a["end"] <= b["start"] for a, b in zip(dev, dev[1:]))
    assert max(x["end"] for x in recs) == r["makespan"]
    c = tmp_path / "dp.csv"
    T.write_csv(c, recs)
    rows = list(csv.DictReader(open(c)))
    assert rows[0].keys() == {"device", "kind", "chunk", "mb", "start", "end", "phase", "route"}


def _summary(orc, policy, P, M, v=1):
    r = orc.evaluate(policy, P, M, v, 1, 2, 1)
    return T.phase_summary(T.records(r["start"], r["end"], _packed(r["kind"], r["chunk"], r["mb"]))), r


def test_phases_1f1b_and_gpipe(orc):
    """1F1B device k: P-k forwards of warmup ("1F1B" §3.1, the pages' count
    before the first backward), then 2(M-P+k) steady ops, then P-k backwards
    of cooldown; with M < P-k the warmup is all M forwards and nothing is
    steady.  GPipe: every forward warmup, every backward cooldown."""
    for P, M in ((4, 8), (8, 16), (5, 3)):
        summ, _ = _summary(orc, "1f1b", P, M)
        for row in summ:
            k, w = row["device"], min(P - row["device"], M)
            assert (row["warmup"]["ops"], row["steady"]["ops"], row["cooldown"]["ops"]) == (w, 2 * (M - w), w)
            # the warmup runs first, the cooldown last, without overlap
            if row["steady"]["ops"]:
                assert row["warmup"]["end"] <= row["steady"]["start"]
                assert row["steady"]["end"] <= row["cooldown"]["start"]
            assert row["warmup"]["busy"] == w * 1 and row["cooldown"]["busy"] == w * 2
        summ, _ = _summary(orc, "gpipe", P, M)
        assert all((x["warmup"]["ops"], x["steady"]["ops"], x["cooldown"]["ops"]) == (M, 0, M) for x in summ)


def test_phases_interleaved(orc):
    """Interleaved 1F1B (reading R4): device k runs min(vP + P - 1 - 2k, vM)
    forwards before its first backward, so that is its warmup."""
    for P, M, v in ((4, 8, 2), (4, 4, 3), (8, 16, 2)):
        summ, _ = _summary(orc, "interleaved", P, M, v)
        for row in summ:
            k = row["device"]
            w = min(v * P + P - 1 - 2 * k, v * M)
            assert row["warmup"]["ops"] == w
            assert row["warmup"]["ops"] + row["steady"]["ops"] + row["cooldown"]["ops"] == 2 * M * v


def test_phases_zero_bubble_and_dualpipe(orc):
    """Zero Bubble with free W keeps 1F1B's F/B order, so its warmup is 1F1B's;
    every W falls after the warmup.  DualPipe: phases cover every op."""
    P, M = 4, 8
    r = orc.zb_evaluate("zb1p", P, M, 1, 2, 0)
    summ = T.phase_summary(T.records(r["start"], r["end"], zb=True))
    for row in summ:
        assert row["warmup"]["ops"] == min(P - row["device"], M)
    recs = T.records(r["start"], r["end"], zb=True)
    assert all(x["phase"] != "warmup" for x in recs if x["kind"] == "W")
    rng = np.random.default_rng(4)
    d = orc.dp_evaluate(P, 4, 4, rng.integers(1, 5, (P, 8)), rng.integers(1, 5, (P, 8)), rng.integers(0, 3, P - 1))
    summ = T.phase_summary(T.records(d["start"], d["end"], dualpipe_m_a=4))
    assert sum(x[ph]["ops"] for x in summ for ph in ("warmup", "steady", "cooldown")) == 2 * P * 8
