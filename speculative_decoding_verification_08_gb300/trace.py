"""Summary of a trace build's timeline of the item kernel (host-side
analysis of the records sv_trace_read returns; nothing here runs on the GPU).

A record is two uint64 words: %globaltimer in ns, and the event word (event
id in bits 56..63, CTA in bits 32..55, the event's argument in bits 0..31).
"""
from __future__ import annotations

TRACE_EVENTS = ("cta_begin", "item_begin", "stage", "item_issued", "item_retired",
                "decide_begin", "decide_end", "producer_end")


def summary(records) -> dict:
    """Where one traced launch's time went, in microseconds from the earliest
    CTA start: the spread of CTA starts, each CTA's delay to its first stage,
    the last stage issued, the last item retired, the last decision written,
    decision times, and items and stages per CTA."""
    import numpy as np
    rec = np.asarray(records, dtype=np.uint64).reshape(-1, 2)
    if rec.shape[0] == 0:
        return {}
    t = rec[:, 0].astype(np.int64)
    w = rec[:, 1]
    ev = (w >> np.uint64(56)).astype(np.int64)
    cta = ((w >> np.uint64(32)) & np.uint64(0xFFFFFF)).astype(np.int64)
    arg = (w & np.uint64(0xFFFFFFFF)).astype(np.int64)
    begin = ev == TRACE_EVENTS.index("cta_begin")
    t0 = t[begin].min() if begin.any() else t.min()
    us = (t - t0) / 1e3

    def last(name):
        m = ev == TRACE_EVENTS.index(name)
        return float(us[m].max()) if m.any() else None

    first_stage = []
    stage = ev == TRACE_EVENTS.index("stage")
    for c in np.unique(cta[begin]):
        mine = stage & (cta == c)
        if mine.any():
            first_stage.append(float(us[mine].min() - us[begin & (cta == c)].min()))
    starts = {}
    decide = []
    for i in np.nonzero(ev == TRACE_EVENTS.index("decide_begin"))[0]:
        starts[(int(cta[i]), int(arg[i]))] = us[i]
    for i in np.nonzero(ev == TRACE_EVENTS.index("decide_end"))[0]:
        s0 = starts.get((int(cta[i]), int(arg[i])))
        if s0 is not None:
            decide.append(float(us[i] - s0))
    items = np.bincount(cta[ev == TRACE_EVENTS.index("item_begin")])
    items = items[items > 0]

    def stats(x):
        return {"median": float(np.median(x)), "max": float(np.max(x))} if len(x) else None

    return {
        "ctas": int(np.unique(cta[begin]).size),
        "cta_begin_spread_us": float(us[begin].max()) if begin.any() else None,
        "first_stage_after_begin_us": stats(first_stage),
        "last_stage_us": last("stage"),
        "last_item_retired_us": last("item_retired"),
        "last_decide_end_us": last("decide_end"),
        "span_us": float(us.max()),
        "decide_us": stats(decide),
        "items_per_cta": stats(items) if items.size else None,
        "stages": int(stage.sum()),
    }
