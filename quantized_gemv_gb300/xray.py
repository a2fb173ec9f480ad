"""X-ray analyser: turns the decode kernel's per-CTA stamps into where one token's time went.

The kernel (built with MK_FLAG_XRAY) has lane 0 of warp 0 of every CTA record {%globaltimer,
clock64, %smid, phase, kind} at the start and end of each phase and of each wait for another
CTA's data (the stamp scheme of the X-ray milestone, monolith page, "M2: X-ray"). %globaltimer is
one clock for the whole GPU, so records of different SMs are aligned by construction; clock64
is per SM and is only used to check the globaltimer's granularity.

The split follows the page's budget bar ("where the time goes", monolith page, "What the demo
looks like"): weight reads (the dequant-GEMV phases), barrier wait (waits on other CTAs' data),
attention, the LM head, and idle (a CTA's time after its own last stamp until the last CTA
finishes).
"""
from __future__ import annotations

import gzip
import json

import numpy as np

PHASE_NAMES = {0: "qkv", 1: "attention", 2: "o_proj", 3: "gate_up", 4: "down", 5: "lm_head", 6: "embed"}
GEMV_PHASES = (0, 2, 3, 4)
KIND_BEGIN, KIND_END, KIND_WAIT_BEGIN, KIND_WAIT_END, KIND_MARK, KIND_STOP = 0, 1, 2, 3, 4, 255


def records(trace: np.ndarray):
    """Yield (cta, [(t_ns, phase, kind), ...]) for every CTA that wrote records (phase and wait
    stamps; sub-phase marks, which carry only the SM clock, are left out).

    Most stamps carry only the SM clock (their %globaltimer field is 0; the kernel reads the global
    timer only at the embedding, at the start of each layer's wait for the previous layer's output
    and at the end of the LM head): their global time is interpolated linearly in clock64 between
    the CTA's neighbouring stamps that carry both, which is exact while the SM clock holds still
    between them."""
    for cta in range(trace.shape[0]):
        rows = trace[cta]
        ends = np.flatnonzero((rows["kind"] == KIND_STOP) | ((rows["gtime"] == 0) & (rows["clk"] == 0)))
        rs = rows[: ends[0]] if len(ends) else rows
        rs = rs[rs["kind"] != KIND_MARK]
        if len(rs) == 0:
            continue
        g = rs["gtime"].astype(np.float64)
        c = rs["clk"].astype(np.float64)
        full = g != 0
        if full.any() and not full.all():
            if full.sum() >= 2:
                g[~full] = np.interp(c[~full], c[full], g[full])
            else:
                g[~full] = g[full][0]
        yield cta, [(int(round(t)), int(ph), int(k)) for t, ph, k in zip(g, rs["phase"], rs["kind"])]


def analyze(trace: np.ndarray, bytes_by_phase: dict | None = None) -> dict:
    """Per-token split of time (ns), averaged over CTAs, plus the critical-path length.

    bytes_by_phase (optional): algorithmic bytes read per phase name over the whole token, used to
    report the bandwidth each phase achieved over its mean active time.
    """
    per_cta = {}
    t_first, t_last = None, None
    for cta, recs in records(trace):
        t_first = recs[0][0] if t_first is None else min(t_first, recs[0][0])
        t_last = recs[-1][0] if t_last is None else max(t_last, recs[-1][0])
        per_cta[cta] = recs
    if not per_cta:
        return {"ctas": 0}
    token_ns = t_last - t_first
    acc = {"weight_read": [], "barrier_wait": [], "attention": [], "lm_head": [], "idle": [], "other": []}
    phase_active = {name: [] for name in PHASE_NAMES.values()}
    for cta, recs in per_cta.items():
        wait = 0
        open_phase, open_wait = {}, None
        active = {name: 0 for name in PHASE_NAMES.values()}
        att_wait = 0
        for t, ph, kind in recs:
            if kind == KIND_BEGIN:
                open_phase[ph] = t
            elif kind == KIND_END and ph in open_phase:
                active[PHASE_NAMES[ph]] += t - open_phase.pop(ph)
            elif kind == KIND_WAIT_BEGIN:
                open_wait = t
            elif kind == KIND_WAIT_END and open_wait is not None:
                wait += t - open_wait
                if 1 in open_phase:  # a wait inside the attention phase (for q/k/v)
                    att_wait += t - open_wait
                open_wait = None
        weight = sum(active[PHASE_NAMES[p]] for p in GEMV_PHASES)
        attention = active["attention"] - att_wait
        head = active["lm_head"]
        idle = t_last - recs[-1][0]
        total = recs[-1][0] - t_first
        acc["weight_read"].append(weight)
        acc["barrier_wait"].append(wait)
        acc["attention"].append(attention)
        acc["lm_head"].append(head)
        acc["idle"].append(idle)
        acc["other"].append(total - weight - wait - attention - head)
        for name, v in active.items():
            phase_active[name].append(v)
    out = {"ctas": len(per_cta), "token_ns": int(token_ns)}
    for k, v in acc.items():
        out[k + "_ns"] = float(np.mean(v))
    out["barrier_wait_share"] = out["barrier_wait_ns"] / token_ns if token_ns else 0.0
    out["phase_mean_ns"] = {k: float(np.mean(v)) for k, v in phase_active.items() if v}
    if bytes_by_phase:
        out["phase_gbs"] = {k: (bytes_by_phase[k] / out["phase_mean_ns"][k]) for k in bytes_by_phase
                            if out["phase_mean_ns"].get(k)}
    return out


def layer_timeline(trace: np.ndarray) -> list:
    """Per-layer wall time (ns) on the critical path: the spread between consecutive moments at
    which the last CTA finished its down_proj phase."""
    ends = {}
    for cta, recs in records(trace):
        k = 0
        for t, ph, kind in recs:
            if ph == 4 and kind == KIND_END:
                ends.setdefault(k, []).append(t)
                k += 1
    last = [max(ends[k]) for k in sorted(ends)]
    return [int(b - a) for a, b in zip(last[:-1], last[1:])]


def export_json(trace: np.ndarray, path: str, meta: dict | None = None):
    """Compact JSON of one token's trace: one list of [t_ns, phase, kind] per CTA (t from token start),
    gzip-compressed when the path ends in .gz."""
    per = dict(records(trace))
    t0 = min(r[0][0] for r in per.values())
    doc = {"meta": meta or {}, "phases": PHASE_NAMES,
           "ctas": {str(c): [[t - t0, ph, k] for t, ph, k in recs] for c, recs in per.items()}}
    text = json.dumps(doc, separators=(",", ":"))
    if path.endswith(".gz"):
        with gzip.open(path, "wt") as f:
            f.write(text)
    else:
        with open(path, "w") as f:
            f.write(text)


def load_json(path: str) -> dict:
    """Read back what export_json wrote."""
    opener = gzip.open if path.endswith(".gz") else open
    with opener(path, "rt") as f:
        return json.load(f)


def critical_path(trace: np.ndarray) -> dict:
    """Per layer, where the dependent chain spends its time (ns, means over layers 1..L-2 so that
    the first and last layers' set-up and tail do not distort them).

    For each GEMV phase P of a layer: `phase_<P>` is the span from the last CTA's end of waiting for
    P's input to the last CTA's end of P (the phase on the critical path); `exchange_<P>` is the span
    from the last CTA's end of the phase that produces P's input to the first and the last CTA's end
    of waiting for it (hop, polling and staging; the two ends bound the spread between CTAs). The
    attention of a layer sits inside `exchange_o_proj`, since o_proj waits for its outputs.
    """
    prev_of = {0: 4, 2: 0, 3: 2, 4: 3}  # producing phase of each GEMV phase's input (QKV <- down)
    ends = {}      # (layer, phase) -> list of end times
    waits = {}     # (layer, consumer phase) -> list of wait-end times
    for _, recs in records(trace):
        layer, open_wait_for = 0, None
        for t, ph, kind in recs:
            if kind == KIND_END and ph in (0, 2, 3, 4):
                ends.setdefault((layer, ph), []).append(t)
                if ph == 4:
                    layer += 1
            elif kind == KIND_WAIT_END and ph in (1, 2, 3, 4):
                # a wait is stamped with the phase that produces the input: 1 -> o_proj, 2 -> gate_up,
                # 3 -> down, 4 -> the next layer's QKV (or the LM head)
                consumer = {1: 2, 2: 3, 3: 4, 4: 0}[ph]
                waits.setdefault((layer, consumer), []).append(t)
    n_layers = max((l for (l, p) in ends if p == 4), default=-1) + 1
    acc = {}
    for l in range(1, n_layers - 1):
        for ph, name in ((0, "qkv"), (2, "o_proj"), (3, "gate_up"), (4, "down")):
            w = waits.get((l, ph))
            e = ends.get((l, ph))
            src = ends.get((l - 1 if ph == 0 else l, prev_of[ph]))
            if not w or not e or not src:
                continue
            acc.setdefault("phase_" + name, []).append(max(e) - max(w))
            acc.setdefault("exchange_" + name + "_first", []).append(min(w) - max(src))
            acc.setdefault("exchange_" + name + "_last", []).append(max(w) - max(src))
    out = {k: float(np.mean(v)) for k, v in acc.items()}
    lt = layer_timeline(trace)
    out["layer"] = float(np.mean(lt[1:-1])) if len(lt) > 2 else (float(np.mean(lt)) if lt else 0.0)
    out["layers"] = n_layers
    return out
