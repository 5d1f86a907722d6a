"""Per-op timeline export: one schedule instance's op times as records, a
Chrome trace (the JSON "traceEvents" format that chrome://tracing and
Perfetto open) or CSV.

The times come from the library (op_start / op_end of pp_sched_eval,
pp_sched_eval_zb or pp_sched_eval_dualpipe); this module only formats them.
Each record is one op: device, kind ("F", "B" or, for Zero Bubble, "W"),
chunk, microbatch, start and end tick, and for DualPipe the route ("A" enters
at device 0, "B" at device P-1).
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
    out.sort(key=lambda r: (r["device"], r["start"], r["end"]))
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
                       "args": {"chunk": r["chunk"], "mb": r["mb"], "start": r["start"], "end": r["end"]}})
    return {"traceEvents": events, "displayTimeUnit": "ms"}


def write_chrome_trace(path, recs, us_per_tick=1.0, name="schedule"):
    with open(path, "w") as f:
        json.dump(chrome_trace(recs, us_per_tick, name), f)


def write_csv(path, recs):
    fields = ["device", "kind", "chunk", "mb", "start", "end"] + (["route"] if recs and "route" in recs[0] else [])
    with open(path, "w", newline="") as f:
        w = csv.DictWriter(f, fieldnames=fields)
        w.writeheader()
        w.writerows(recs)
