"""Timeline of one traced megakernel launch (see mk_set_trace / mk_get_trace).

Each instruction slot holds %globaltimer stamps (ns): the producer's first
bulk copy of the instruction, the consumers' wait start and end, the end of
the op's prologue phase (norm / split combine), the end of its ring loop and
the body end, and the moment the completion signal (a release reduction)
retired (a missing mid stamp falls back to the previous one).  `summarize` attributes the step's time the way "Megakernels:
Deleting the Kernel Boundary", section "What it buys, and where the time
still goes", breaks down a forward pass: time spent waiting on dependencies
versus time spent in instruction bodies, per opcode and per layer.
`chrome_trace` writes the timeline in Chrome trace-event JSON."""
from __future__ import annotations

import json

import numpy as np

from . import _lib as L


def _rows(trace, queues, n_sm, max_pc):
    t = trace.astype(np.int64)
    base = None
    rows = []
    for s in range(n_sm):
        for pc in range(max_pc):
            I = queues[s * max_pc + pc]
            if I.op == 0:
                break
            ts = t[s, pc]
            if ts[1] == 0 or ts[5] == 0:
                continue
            m0 = ts[3] if ts[3] >= ts[2] else ts[2]
            m1 = ts[4] if ts[4] >= m0 else m0
            rows.append((s, pc, I.op, I.layer, ts[0], ts[1], ts[2], ts[5], m0, m1, ts[6],
                         ts[7] if ts[7] >= ts[5] else ts[5]))
            base = ts[1] if base is None else min(base, ts[1])
    return rows, base


# Consecutive phases of a layer (the split MLP; a fused MLP shows up as MLP).
_CHAIN = ("QKV", "ATTN", "OPROJ", "MLP_UP", "MLP_DOWN")


def _hops(rows) -> dict:
    """Per dependency hop, averaged over the inner layers: from the moment
    the producing phase's last instruction ended its body to the end of the
    consuming instructions' prologues (min / median / max over the
    consumers), and the consumers' median time from prologue end to body
    end.  The hop covers the producer's completion signal, its propagation,
    the consumer's wait and the loading of the phase's input vector."""
    by = {}
    for s, pc, op, layer, tp, tw0, tw1, te, m0, m1, rw, tsig in rows:
        by.setdefault((layer, L.OP_NAMES[op]), []).append((te, m0))
    layers = sorted({k[0] for k in by if k[1] in _CHAIN})
    out = {}
    pairs = [(a, b, 0) for a, b in zip(_CHAIN, _CHAIN[1:])] + [(_CHAIN[-1], _CHAIN[0], 1)]
    for a, b, dl in pairs:
        lat, body = [], []
        for l in layers[1:-1]:
            pa, pb = by.get((l, a)), by.get((l + dl, b))
            if not pa or not pb:
                continue
            last = max(t for t, _ in pa)
            pe = np.array([m for _, m in pb], dtype=np.float64)
            lat.append(((pe.min() - last), np.median(pe) - last, pe.max() - last))
            body.append(float(np.median([t - m for t, m in pb])))
        if lat:
            v = np.array(lat).mean(axis=0) / 1e3
            out[f"{a}->{b}"] = {"min_us": float(v[0]), "median_us": float(v[1]),
                                "max_us": float(v[2]),
                                "consumer_ring_and_epilogue_us": float(np.mean(body)) / 1e3}
    return out


def summarize(trace, queues, n_sm: int, max_pc: int) -> dict:
    rows, base = _rows(trace, queues, n_sm, max_pc)
    if not rows:
        return {}
    end = max(r[7] for r in rows)
    by_op = {}
    for s, pc, op, layer, tp, tw0, tw1, te, m0, m1, rw, tsig in rows:
        d = by_op.setdefault(L.OP_NAMES[op], {"n": 0, "wait_us": 0.0, "body_us": 0.0,
                                               "max_wait_us": 0.0, "prologue_us": 0.0,
                                               "ring_us": 0.0, "epilogue_us": 0.0,
                                               "ring_data_wait_us": 0.0})
        d["ring_data_wait_us"] += rw / 1e3
        d["n"] += 1
        d["wait_us"] += (tw1 - tw0) / 1e3
        d["body_us"] += (te - tw1) / 1e3
        d["prologue_us"] += (m0 - tw1) / 1e3
        d["ring_us"] += (m1 - m0) / 1e3
        d["epilogue_us"] += (te - m1) / 1e3
        d["max_wait_us"] = max(d["max_wait_us"], (tw1 - tw0) / 1e3)
    for d in by_op.values():
        for k in ("wait", "body", "prologue", "ring", "epilogue", "ring_data_wait"):
            d[f"mean_{k}_us"] = d[f"{k}_us"] / d["n"]
    # per layer and phase: when the last instruction of the phase finished
    phase_end = {}
    for s, pc, op, layer, tp, tw0, tw1, te, m0, m1, rw, tsig in rows:
        k = (layer, L.OP_NAMES[op])
        phase_end[k] = max(phase_end.get(k, 0), te - base)
    layers = sorted({k[0] for k in phase_end})
    per_layer = []
    prev = 0
    for l in layers:
        e = max(v for k, v in phase_end.items() if k[0] == l)
        per_layer.append({"layer": l, "end_us": e / 1e3, "span_us": (e - prev) / 1e3,
                          "phases_end_us": {k[1]: v / 1e3 for k, v in phase_end.items()
                                            if k[0] == l}})
        prev = e
    busy = np.zeros(n_sm)
    waited = np.zeros(n_sm)
    for s, pc, op, layer, tp, tw0, tw1, te, m0, m1, rw, tsig in rows:
        busy[s] += te - tw1
        waited[s] += tw1 - tw0
    return {"step_us": (end - base) / 1e3, "by_op": by_op, "per_layer": per_layer,
            "hops": _hops(rows),
            "mean_sm_body_us": float(busy.mean() / 1e3),
            "mean_sm_wait_us": float(waited.mean() / 1e3)}


def chrome_trace(trace, queues, n_sm: int, max_pc: int, path: str):
    rows, base = _rows(trace, queues, n_sm, max_pc)
    ev = []
    for s, pc, op, layer, tp, tw0, tw1, te, m0, m1, rw, tsig in rows:
        name = f"{L.OP_NAMES[op]} L{layer}"
        ev.append({"name": "wait " + name, "ph": "X", "pid": 0, "tid": s,
                   "ts": (tw0 - base) / 1e3, "dur": (tw1 - tw0) / 1e3})
        ev.append({"name": name, "ph": "X", "pid": 0, "tid": s, "ts": (tw1 - base) / 1e3,
                   "dur": (te - tw1) / 1e3,
                   "args": {"prologue_end": (m0 - base) / 1e3, "ring_end": (m1 - base) / 1e3,
                            "signal_done": (tsig - base) / 1e3,
                            "ring_data_wait_us": rw / 1e3}})
        if tp:
            ev.append({"name": "issue " + name, "ph": "i", "pid": 1, "tid": s,
                       "ts": (tp - base) / 1e3, "s": "t"})
    with open(path, "w") as f:
        json.dump({"traceEvents": ev}, f)
