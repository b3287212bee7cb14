"""Summary of a trace build's timeline of the item kernel (host-side
analysis of the records sv_trace_read returns; nothing here runs on the GPU).

A record is two uint64 words: %globaltimer in ns, and the event word (event
id in bits 56..63, CTA in bits 32..55, the event's argument in bits 0..31).
Consecutive launches append to each CTA's region in order, each launch's
records of a CTA opening with its "cta_placed" record.
"""
from __future__ import annotations

TRACE_EVENTS = ("cta_begin", "item_begin", "stage", "item_issued", "item_retired",
                "decide_begin", "decide_end", "producer_end", "cta_placed", "cta_end",
                # sampling from logits (bulk-copy workers)
                "lg_claim", "lg_ready", "lg_issued", "lg_chunk_done", "lg_decide", "lg_last", "lg_merged")


def _fields(records):
    import numpy as np
    rec = np.asarray(records, dtype=np.uint64).reshape(-1, 2)
    t = rec[:, 0].astype(np.int64)
    w = rec[:, 1]
    ev = (w >> np.uint64(56)).astype(np.int64)
    cta = ((w >> np.uint64(32)) & np.uint64(0xFFFFFF)).astype(np.int64)
    arg = (w & np.uint64(0xFFFFFFFF)).astype(np.int64)
    return rec, t, ev, cta, arg


def split_launches(records):
    """The records of each traced launch, in launch order.  Records are in
    slot order within each CTA's region; a CTA's "cta_placed" record opens
    its part of the next launch.  Records without any placement record are
    one launch."""
    import numpy as np
    rec, t, ev, cta, arg = _fields(records)
    if rec.shape[0] == 0:
        return []
    placed = ev == TRACE_EVENTS.index("cta_placed")
    if not placed.any():
        return [rec]
    launch = np.zeros(rec.shape[0], dtype=np.int64)
    for c in np.unique(cta):
        idx = np.nonzero(cta == c)[0]           # this CTA's records, in slot order
        launch[idx] = np.cumsum(placed[idx]) - 1
    keep = launch >= 0
    return [rec[keep & (launch == k)] for k in range(int(launch.max()) + 1)]


def summary(records) -> dict:
    """Where one traced launch's time went, in microseconds from the earliest
    CTA start: the spread of CTA starts, each CTA's delay to its first stage,
    the last stage issued, the last item retired, the last decision written,
    decision times, and items and stages per CTA (plus, when the records
    carry them, each CTA's last retirement, producer end and exit)."""
    import numpy as np
    rec, t, ev, cta, arg = _fields(records)
    if rec.shape[0] == 0:
        return {}
    begin = ev == TRACE_EVENTS.index("cta_begin")
    t0 = t[begin].min() if begin.any() else t.min()
    us = (t - t0) / 1e3

    def last(name):
        m = ev == TRACE_EVENTS.index(name)
        return float(us[m].max()) if m.any() else None

    def stats(x):
        return {"median": float(np.median(x)), "max": float(np.max(x))} if len(x) else None

    def per_cta_last(name):
        m = ev == TRACE_EVENTS.index(name)
        return [float(us[m & (cta == c)].max()) for c in np.unique(cta[m])]

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

    out = {
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
    placed = ev == TRACE_EVENTS.index("cta_placed")
    if placed.any():
        out["cta_placed_us"] = stats(us[placed])           # negative: before the first start
        out["cta_last_stage_us"] = stats(per_cta_last("stage"))
        out["cta_last_retired_us"] = stats(per_cta_last("item_retired"))
        out["cta_producer_end_us"] = stats(per_cta_last("producer_end"))
        out["cta_end_us"] = stats(per_cta_last("cta_end"))
    return out


def timeline(records) -> dict:
    """Every traced launch's summary, and between consecutive launches: the
    period from one launch's first CTA start to the next one's, how long
    before the previous grid's last CTA exit the next grid's CTAs were placed
    (median), and the gap from that exit to the next grid's first start
    (which includes the previous grid's completion and the dependent wait)."""
    import numpy as np
    parts = split_launches(records)
    launches = [summary(r) for r in parts]
    between = []
    for a, b in zip(parts, parts[1:]):
        _, ta, eva, _, _ = _fields(a)
        _, tb, evb, _, _ = _fields(b)
        ia, ib = TRACE_EVENTS.index("cta_begin"), TRACE_EVENTS.index("cta_end")
        pl = TRACE_EVENTS.index("cta_placed")
        if not ((eva == ia).any() and (evb == ia).any() and (eva == ib).any()):
            continue
        a_begin, b_begin = ta[eva == ia].min(), tb[evb == ia].min()
        a_end = ta[eva == ib].max()
        between.append({
            "period_us": float(b_begin - a_begin) / 1e3,
            "placed_before_prev_exit_us": float(a_end - np.median(tb[evb == pl])) / 1e3
            if (evb == pl).any() else None,
            "prev_exit_to_start_us": float(b_begin - a_end) / 1e3,
        })
    return {"launches": launches, "between": between}
