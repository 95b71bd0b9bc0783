"""Intra-kernel event traces (HGEMM_OPT_TRACE) -> summaries and Chrome traces.

The kernels append (time, CTA, role, kind, tile, value) records when a
handle's trace buffer is on; see hgemm_trace_record_t in include/hgemm.h.
``chrome_trace`` turns them into the Trace Event Format that Perfetto and
chrome://tracing open (one process per CTA, one thread per role), the same
kind of timeline the tcgen05 walkthrough builds from clock-register stamps.
"""
from __future__ import annotations

import collections
import json

ROLES = {0: "cta", 1: "tma", 2: "mma", 3: "epilogue"}
KINDS = {1: "kernel_begin", 2: "kernel_end", 3: "item_begin", 4: "item_end", 5: "partial_stored", 6: "reduced",
         7: "stall_cycles"}


def spans(rows):
    """Pairs item begin/end per (cta, role) in time order -> list of dicts."""
    by = collections.defaultdict(list)
    for t, cta, role, kind, item, value in rows:
        by[(cta, role)].append((t, kind, item, value))
    out = []
    for (cta, role), ev in by.items():
        ev.sort()
        open_ = None
        for t, kind, item, value in ev:
            if kind == 3:
                open_ = (t, item, value)
            elif kind == 4 and open_ is not None:
                out.append(dict(cta=cta, role=ROLES.get(role, str(role)), tile=open_[1], t0=open_[0], t1=t,
                                begin_value=open_[2], end_value=value))
                open_ = None
    return out


def launch_clocks(rows):
    """SM clock (MHz) of every CTA launch in the records: each CTA's kernel
    begin and end records, paired in time order, carry the global timer (ns)
    and the low 31 bits of the SM cycle counter, so cycles / ns over the
    pair is the clock that CTA ran at.  Works for records of many launches
    (HGEMM_OPT_TRACE_ITEMS = 0 keeps only these records)."""
    by = collections.defaultdict(list)
    for t, cta, role, kind, item, value in rows:
        if role == 0 and kind in (1, 2):
            by[cta].append((t, kind, value))
    out = []
    for ev in by.values():
        ev.sort()
        begin = None
        for t, kind, value in ev:
            if kind == 1:
                begin = (t, value)
            elif begin is not None:
                if t > begin[0]:
                    out.append(((value - begin[1]) % (1 << 31)) / (t - begin[0]) * 1e3)
                begin = None
    return out


def summary(rows):
    """Kernel span, per-role busy time and the spread of CTA end times (ns)."""
    if not rows:
        return {}
    t0 = min(r[0] for r in rows)
    begins = [r[0] - t0 for r in rows if r[3] == 1]
    ends = [r[0] - t0 for r in rows if r[3] == 2]
    sp = spans(rows)
    busy = collections.defaultdict(int)
    for s in sp:
        busy[s["role"]] += s["t1"] - s["t0"]
    n_cta = max(1, len(begins))
    # SM clock: cycle-counter delta over timer delta between a CTA's begin and end
    be = {}
    for t, cta, role, kind, item, value in rows:
        if kind in (1, 2):
            be.setdefault(cta, {})[kind] = (t, value)
    mhz = [((v[2][1] - v[1][1]) % (1 << 31)) / max(1, v[2][0] - v[1][0]) * 1e3
           for v in be.values() if 1 in v and 2 in v and v[2][0] > v[1][0]]
    stalls = collections.defaultdict(int)
    for r in rows:
        if r[3] == 7:
            stalls[ROLES.get(r[2], str(r[2]))] += r[5]
    return {
        "sm_mhz": sorted(mhz)[len(mhz) // 2] if mhz else None,
        "stall_cycles_per_cta": {k: v / n_cta for k, v in stalls.items()},
        "span_ns": max(r[0] for r in rows) - t0,
        "cta_begin_ns": [min(begins), max(begins)] if begins else None,
        "cta_end_ns": [min(ends), max(ends)] if ends else None,
        "busy_ns_per_cta": {k: v / n_cta for k, v in busy.items()},
        "items": len(sp),
        "partials": sum(1 for r in rows if r[3] == 5),
        "reductions": sum(1 for r in rows if r[3] == 6),
    }


def chrome_trace(rows, path=None):
    """Trace Event Format: complete events per item, instants for the rest."""
    if not rows:
        return {"traceEvents": []}
    t0 = min(r[0] for r in rows)
    ev = []
    for s in spans(rows):
        ev.append({"name": "tile %d" % s["tile"], "ph": "X", "pid": s["cta"], "tid": s["role"],
                   "ts": (s["t0"] - t0) / 1e3, "dur": max(0.001, (s["t1"] - s["t0"]) / 1e3),
                   "args": {"begin": s["begin_value"], "end": s["end_value"]}})
    for t, cta, role, kind, item, value in rows:
        if kind in (1, 2, 5, 6):
            ev.append({"name": KINDS[kind], "ph": "i", "s": "t", "pid": cta, "tid": ROLES.get(role, str(role)),
                       "ts": (t - t0) / 1e3, "args": {"tile": item, "value": value}})
    doc = {"traceEvents": ev, "displayTimeUnit": "ns"}
    if path:
        with open(path, "w") as f:
            json.dump(doc, f)
    return doc
