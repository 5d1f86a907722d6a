"""Per-op timeline export: one schedule instance's op times as records, a
Chrome trace (the JSON "traceEvents" format that chrome://tracing and
Perfetto open) or CSV.

The times come from the library (op_start / op_end of pp_sched_eval,
pp_sched_eval_zb or pp_sched_eval_dualpipe); this module only formats them.
Each record is one op: device, kind ("F", "B" or, for Zero Bubble, "W"),
chunk, microbatch, start and end tick, its phase on the device, and for
DualPipe the route ("A" enters at device 0, "B" at device P-1).

Phases ("1F1B" §3.1's warmup / steady / cooldown, asked per stage by "Pipeline
scheduling" (M040) §09's checklist), read off each device's op order: the
warmup is the run of forwards before the device's first backward (P - k of
them on device k under 1F1B, the pages' count), the cooldown is everything
after its last forward, the steady phase everything between.  GPipe has no
steady phase: all forwards are its warmup, all backwards its cooldown.
"""
from __future__ import annotations

import csv
import json

import numpy as np

KINDS = ("F", "B", "W")


def records(op_start, op_end, ops=None, zb=False, dualpipe_m_a=None):
    """Records of one instance.

    op_start, op_end: [P][O] ticks (pp_sched_eval, O = 2*M*v ops per device,
    in the device's order) with `ops` the plan's packed op words [P][O]
    (binding.Plan.tables()[0]); or, with zb=True, [P][3][M] ticks of
    pp_sched_eval_zb (kind F, B, W; microbatch); or, with dualpipe_m_a set
    (route A's microbatch count), [P][2][M] ticks of pp_sched_eval_dualpipe
    (block, kind F / B, microbatch): block s of microbatch g runs on device s
    for route A (g < m_a) and on device P-1-s for route B."""
    st = np.asarray(op_start)
    en = np.asarray(op_end)
    out = []
    if dualpipe_m_a is not None:
        P, _, M = st.shape
        for s in range(P):
            for kd in range(2):
                for g in range(M):
                    a = g < dualpipe_m_a
                    out.append(dict(device=s if a else P - 1 - s, kind=KINDS[kd], chunk=0, mb=g,
                                    start=int(st[s, kd, g]), end=int(en[s, kd, g]), route="A" if a else "B"))
    elif zb:
        P, _, M = st.shape
        for k in range(P):
            for kd in range(3):
                for m in range(M):
                    out.append(dict(device=k, kind=KINDS[kd], chunk=0, mb=m, start=int(st[k, kd, m]),
                                    end=int(en[k, kd, m])))
    else:
        ops = np.asarray(ops).astype(np.int64)
        P, O = st.shape
        for k in range(P):
            for j in range(O):
                w = int(ops[k, j])
                out.append(dict(device=k, kind=KINDS[(w >> 31) & 1], chunk=(w >> 24) & 0x7F, mb=w & 0xFFFFFF,
                                start=int(st[k, j]), end=int(en[k, j])))
    if dualpipe_m_a is not None or zb:
        # no plan order: a device's order is its time order (F and B take at
        # least one tick, so they never tie; a W never precedes its B)
        out.sort(key=lambda r: (r["device"], r["start"], r["end"]))
        _label_phases(out)
    else:
        _label_phases(out)  # plan order: records were built device by device in op order
        out.sort(key=lambda r: (r["device"], r["start"], r["end"]))
    return out


def _label_phases(recs):
    """Add each record's phase; `recs` lists each device's ops contiguously in
    the device's order."""
    by_dev = {}
    for r in recs:
        by_dev.setdefault(r["device"], []).append(r)
    for dev in by_dev.values():
        kinds = [r["kind"] for r in dev]
        first_b = kinds.index("B") if "B" in kinds else len(kinds)
        last_f = len(kinds) - 1 - kinds[::-1].index("F") if "F" in kinds else -1
        for i, r in enumerate(dev):
            r["phase"] = "warmup" if i < first_b else ("cooldown" if i > last_f else "steady")


def phase_summary(recs):
    """Per device and phase: op count, first start and last end tick (None
    for an empty phase), and busy ticks."""
    out = []
    for k in sorted({r["device"] for r in recs}):
        row = {"device": k}
        for ph in ("warmup", "steady", "cooldown"):
            rs = [r for r in recs if r["device"] == k and r["phase"] == ph]
            row[ph] = {"ops": len(rs), "start": min((r["start"] for r in rs), default=None),
                       "end": max((r["end"] for r in rs), default=None),
                       "busy": sum(r["end"] - r["start"] for r in rs)}
        out.append(row)
    return out


def chrome_trace(recs, us_per_tick=1.0, name="schedule"):
    """Chrome trace dict: one complete event ("ph": "X") per op, one thread
    row per device."""
    events = [{"name": "process_name", "ph": "M", "pid": 0, "args": {"name": name}}]
    for k in sorted({r["device"] for r in recs}):
        events.append({"name": "thread_name", "ph": "M", "pid": 0, "tid": k, "args": {"name": f"device {k}"}})
    for r in recs:
        label = f"{r['kind']}{r['mb']}" + (f".c{r['chunk']}" if r["chunk"] else "") + \
            (f".{r['route']}" if "route" in r else "")
        events.append({"name": label, "cat": r["kind"], "ph": "X", "pid": 0, "tid": r["device"],
                       "ts": r["start"] * us_per_tick, "dur": (r["end"] - r["start"]) * us_per_tick,
                       "args": {"chunk": r["chunk"], "mb": r["mb"], "start": r["start"], "end": r["end"],
                                "phase": r["phase"]}})
    return {"traceEvents": events, "displayTimeUnit": "ms"}


def write_chrome_trace(path, recs, us_per_tick=1.0, name="schedule"):
    with open(path, "w") as f:
        json.dump(chrome_trace(recs, us_per_tick, name), f)


def write_csv(path, recs):
    fields = ["device", "kind", "chunk", "mb", "start", "end", "phase"] + \
        (["route"] if recs and "route" in recs[0] else [])
    with open(path, "w", newline="") as f:
        w = csv.DictWriter(f, fieldnames=fields)
        w.writeheader()
        w.writerows(recs)
