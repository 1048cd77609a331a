"""Reads the per-work-item trace of a decode step (schedule built with
trace=1) and summarises it: where each SM's time went, per opcode and per
layer, and the producer/consumer stall counters.  Can also write a Chrome
trace (one row per SM), the timeline view of the pages' per-SM figures."""
from __future__ import annotations

import json

import numpy as np

from . import OPS

WORK_OPS = {32: "ATTN_SLICE", 33: "MOE_UP_TILE", 34: "MOE_DOWN_TILE", 35: "CLAIM_END", 36: "EXIT"}


def op_name(op: int) -> str:
    return OPS.get(op, WORK_OPS.get(op, str(op)))


def read(session) -> dict:
    import torch
    s = session.sched
    nsm = s.num_sms
    st = session.region("stats", torch.int64, nsm * 8).view(nsm, 8).cpu().numpy()
    total = session.sched.workspace_offset("stats") - session.sched.workspace_offset("trace")
    cap = total // (nsm * 4 * 8)
    tr = session.region("trace", torch.int64, nsm * cap * 4).view(nsm, cap, 4).cpu().numpy()
    recs = []
    for sm in range(nsm):
        n = int(min(st[sm, 3], cap))
        for r in tr[sm, :n]:
            tag = int(r[3])
            recs.append((sm, int(r[0]), int(r[1]), int(r[2]), tag & 0xff, (tag >> 8) & 0xff,
                         (tag >> 16) & 0xffffff, (tag >> 40) & 0xffffff))
    a = np.array(recs, dtype=np.int64).reshape(-1, 8)
    return {"rec": a, "stats": st, "num_sms": nsm}


def summary(t: dict) -> str:
    a, st = t["rec"], t["stats"]
    if a.size == 0:
        return "empty trace"
    t0 = a[:, 1].min()
    span = (a[:, 3].max() - t0) / 1e3
    lines = [f"step span {span:.1f} us over {t['num_sms']} SMs, {len(a)} work items"]
    lines.append(f"{'op':>22} {'items':>7} {'busy us/SM':>11} {'wait us/SM':>11} {'mean busy us':>13}")
    nsm = t["num_sms"]
    for op in sorted(set(a[:, 4].tolist())):
        m = a[:, 4] == op
        busy = (a[m, 3] - a[m, 2]).sum() / 1e3
        wait = (a[m, 2] - a[m, 1]).sum() / 1e3
        lines.append(f"{op_name(op):>22} {m.sum():7d} {busy / nsm:11.2f} {wait / nsm:11.2f} "
                     f"{busy / max(1, m.sum()):13.2f}")
    c = st.astype(np.float64)
    # busy spans an item from its inputs' arrival to its end, stage waits included
    lines.append("per SM mean: consumer wait-on-counters %.1f us, wait-on-stages %.1f us (within busy), "
                 "busy %.1f us, items %.0f" % (c[:, 0].mean() / 1e3, c[:, 1].mean() / 1e3, c[:, 2].mean() / 1e3,
                                               c[:, 3].mean()))
    lines.append("per SM mean: producer wait-on-free-stage %.1f us, wait-on-routing %.1f us, "
                 "wait-on-work-ring %.1f us, claims %.0f" % (c[:, 4].mean() / 1e3, c[:, 5].mean() / 1e3,
                                                             c[:, 6].mean() / 1e3, c[:, 7].mean()))
    # per layer: when its items start and end
    layers = sorted(set(a[:, 5].tolist()))
    lines.append("layer  first-start  last-end  (us from step start)")
    for l in layers[:4] + layers[-2:]:
        m = a[:, 5] == l
        lines.append(f"{l:5d} {(a[m, 1].min() - t0) / 1e3:12.1f} {(a[m, 3].max() - t0) / 1e3:9.1f}")
    return "\n".join(lines)


def phases(t: dict) -> str:
    """The per-layer critical path: for each op of a layer, when its first
    and last items start and when its last item ends, in microseconds from
    the layer's first start, as medians over the middle layers (the first
    two and the last are left out: start-up and the LM head), and the median
    layer period (first start to the next layer's first start)."""
    a = t["rec"]
    if a.size == 0:
        return "empty trace"
    layers = sorted(set(a[:, 5].tolist()))
    mid = layers[2:-2] if len(layers) > 5 else layers
    starts = {l: a[a[:, 5] == l, 2].min() for l in layers}
    rows: dict = {}
    periods = []
    for l in mid:
        m = a[:, 5] == l
        s0 = starts[l]
        if l + 1 in starts:
            periods.append((starts[l + 1] - s0) / 1e3)
        for op in set(a[m, 4].tolist()):
            mo = m & (a[:, 4] == op)
            rows.setdefault(op, []).append((mo.sum(), (a[mo, 2].min() - s0) / 1e3, (a[mo, 2].max() - s0) / 1e3,
                                            (a[mo, 3].max() - s0) / 1e3, np.median(a[mo, 3] - a[mo, 2]) / 1e3))
    lines = [f"layer period (median over layers {mid[0]}..{mid[-1]}): {np.median(periods):.1f} us" if periods
             else "one layer"]
    lines.append(f"{'op':>22} {'items':>6} {'first go':>9} {'last go':>8} {'last end':>9} {'busy p50':>9}")
    order = sorted(rows, key=lambda op: np.median([r[1] for r in rows[op]]))
    for op in order:
        r = np.array(rows[op], dtype=np.float64)
        med = np.median(r, axis=0)
        lines.append(f"{op_name(op):>22} {med[0]:6.0f} {med[1]:9.1f} {med[2]:8.1f} {med[3]:9.1f} {med[4]:9.2f}")
    return "\n".join(lines)


def chrome_trace(t: dict, path: str) -> None:
    a = t["rec"]
    t0 = a[:, 1].min() if a.size else 0
    ev = []
    for sm, tp, tg, te, op, layer, task, a0 in a.tolist():
        ev.append({"name": f"{op_name(op)} L{layer}", "ph": "X", "pid": 0, "tid": sm,
                   "ts": (tg - t0) / 1e3, "dur": max(0.001, (te - tg) / 1e3),
                   "args": {"task": task, "a0": a0, "wait_us": (tg - tp) / 1e3}})
    with open(path, "w") as f:
        json.dump({"traceEvents": ev}, f)
