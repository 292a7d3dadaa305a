"""Timeline of the forward kernel from its traced build (libattn_fwd_trace.so).

    python -m attention_forward_06_gb300.trace --workload train [--launches 4] [--dump-cta C]

runs the workload through the traced library (same results as the default
build, bit for bit), reads the events of the last launch (include/attn_fwd_trace.h)
and prints where the launch's time goes, per CTA and in medians:

    span             first CTA start to last CTA end (the kernel's own extent)
    start_us         launch start (earliest CTA start) to a CTA's first S products
    step_us          interval between consecutive P.V issues of Q tile 0 inside an item
    boundary_us      the extra time between an item's last P.V and the next item's first,
                     beyond one step
    softmax_us       S_t(j) ready to P_t(j) handed over (per Q tile)
    tail_us          spread of the CTAs' end times (with their 10th, 50th and 90th percentiles)
    items_per_cta    work items a CTA processed

The recording adds a global store and a timer read per event, so the figures
run slower than the default build's (the train launch by about a seventh).  A
role keeps its first 2048 events per CTA; for launches longer than that (the
long-context workload) the summary uses the kept events and reports no end
times.
"""
from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np
import torch

from . import _lib
from .inputs import WORKLOADS, draw_workload

REC = np.dtype([("t", "<u8"), ("code", "<u4"), ("arg", "<u4")])
PRODUCER, ISSUER, SOFTMAX0, SOFTMAX1, STORE = range(5)


def read(lib) -> tuple[np.ndarray, np.ndarray]:
    """(counts [ctas, roles], records [ctas, roles, events]) of the launches since the last read."""
    ctas, roles, events = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    lib.attn_fwd_trace_read(None, 0, ctypes.byref(ctas), ctypes.byref(roles), ctypes.byref(events))
    n_bytes = 4 * ctas.value * roles.value
    r_bytes = REC.itemsize * ctas.value * roles.value * events.value
    buf = (ctypes.c_uint8 * (n_bytes + r_bytes))()
    st = lib.attn_fwd_trace_read(buf, n_bytes + r_bytes, None, None, None)
    if st != 0:
        raise RuntimeError(f"attn_fwd_trace_read failed with status {st}")
    raw = np.frombuffer(buf, dtype=np.uint8)
    counts = raw[:n_bytes].view("<u4").reshape(ctas.value, roles.value).copy()
    recs = raw[n_bytes:].view(REC).reshape(ctas.value, roles.value, events.value).copy()
    return counts, recs


def events(counts, recs, cta, role, code=None):
    """Kept events of one role of one CTA (optionally of one code), in order."""
    n = min(int(counts[cta, role]), recs.shape[2])
    e = recs[cta, role, :n]
    return e if code is None else e[e["code"] == code]


def summarize(counts: np.ndarray, recs: np.ndarray) -> dict:
    """The figures listed in the module docstring.  A CTA whose roles reached more events than the buffer keeps
    (long launches) contributes its kept steps and boundaries but no end time (`truncated_ctas` counts them)."""
    ctas = [c for c in range(counts.shape[0]) if counts[c, PRODUCER] > 0]
    if not ctas:
        raise ValueError("no CTA recorded any event")
    starts = np.array([events(counts, recs, c, PRODUCER, 0)["t"][0] for c in ctas], dtype=np.int64)
    complete = [c for c in ctas if len(events(counts, recs, c, ISSUER, 13)) > 0]
    ends = np.array([events(counts, recs, c, ISSUER, 13)["t"][-1] for c in complete], dtype=np.int64)
    t0 = starts.min()
    first_s, steps, bounds, items, softmax = [], [], [], [], []
    for c in ctas:
        iss = events(counts, recs, c, ISSUER)
        items.append(int((iss["code"] == 12).sum()))
        sel = iss[(iss["code"] == 12) | (iss["code"] == 11)]
        if (iss["code"] == 12).any():
            first_s.append(int(iss[iss["code"] == 12]["t"][0]) - int(t0))
        # P.V issue times of Q tile 0, split by item
        per_item, cur = [], []
        for ev in sel:
            if ev["code"] == 12:
                if cur:
                    per_item.append(cur)
                cur = []
            elif ev["arg"] == 0:
                cur.append(int(ev["t"]))
        if cur:
            per_item.append(cur)
        for k, pv in enumerate(per_item):
            steps.extend(np.diff(pv).tolist())
            if k + 1 < len(per_item) and per_item[k + 1]:
                bounds.append(per_item[k + 1][0] - pv[-1])
        for role in (SOFTMAX0, SOFTMAX1):
            sm = events(counts, recs, c, role)
            ready = sm[sm["code"] == 20]["t"].astype(np.int64)
            hand = sm[sm["code"] == 21]["t"].astype(np.int64)
            n = min(len(ready), len(hand))
            softmax.extend((hand[:n] - ready[:n]).tolist())
    step = float(np.median(steps)) if steps else float("nan")
    have_ends = ends.size > 0
    return {
        "ctas": len(ctas),
        "truncated_ctas": len(ctas) - len(complete),
        "span_us": (int(ends.max()) - int(t0)) / 1e3 if have_ends else float("nan"),
        "start_us": float(np.median(first_s)) / 1e3 if first_s else float("nan"),
        "step_us": step / 1e3,
        "steps": len(steps),
        "boundary_us": (float(np.median(bounds)) - step) / 1e3 if bounds else float("nan"),
        "boundaries": len(bounds),
        "softmax_us": float(np.median(softmax)) / 1e3 if softmax else float("nan"),
        "tail_us": (int(ends.max()) - int(ends.min())) / 1e3 if have_ends else float("nan"),
        "cta_end_us_p10_p50_p90": ([float(np.percentile(ends - t0, q)) / 1e3 for q in (10, 50, 90)]
                                   if have_ends else None),
        "items_per_cta": float(np.mean(items)),
    }


NAMES = {0: "cta start", 1: "item published", 2: "K load", 3: "V load", 11: "P.V issued", 12: "item's first S",
         13: "MMAs done", 20: "S ready", 21: "P handed off", 22: "V share converted", 23: "O read", 24: "O staged",
         30: "O store issued", 31: "stores landed"}
ROLE_NAMES = ["producer", "issuer", "softmax0", "softmax1", "store"]


def dump(counts: np.ndarray, recs: np.ndarray, cta: int, t_from_us: float = 0.0, t_to_us: float = 1e9) -> list[str]:
    """One CTA's events of every role merged in time order, as lines 'time_us role event arg' (times from the
    launch's first CTA start)."""
    ctas = [c for c in range(counts.shape[0]) if counts[c, PRODUCER] > 0]
    t0 = min(int(events(counts, recs, c, PRODUCER, 0)["t"][0]) for c in ctas)
    rows = []
    for role in range(counts.shape[1]):
        for ev in events(counts, recs, cta, role):
            t = (int(ev["t"]) - t0) / 1e3
            if t_from_us <= t <= t_to_us:
                arg = int(ev["arg"])
                rows.append((t, f"{t:9.3f} {ROLE_NAMES[role]:9s} {NAMES.get(int(ev['code']), ev['code'])} "
                               f"{arg - (1 << 32) if arg >= 1 << 31 else arg}"))
    return [r for _, r in sorted(rows)]


def run(workload: str, launches: int = 4, dump_cta: int | None = None) -> dict:
    w = WORKLOADS[workload]
    lib = _lib.load("attn_fwd_trace", build_if_missing=True)
    dev = torch.device("cuda", 0)
    q, k, v = [t.to(dev) for t in draw_workload(w)]
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(launches):
        flush.zero_()  # inputs come from HBM, as in the benchmark
        read(lib)  # keep only the last launch
        st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.Hq, w.Hkv,
                          w.Sq, w.Sk, w.D, w.causal, ctypes.c_float(w.scale), stream)
        if st != 0:
            raise RuntimeError(f"attn_fwd failed with status {st}")
    counts, recs = read(lib)
    out = {"workload": w.label(), **summarize(counts, recs)}
    if dump_cta is not None:
        out["events"] = dump(counts, recs, dump_cta)
    return out


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="train", choices=sorted(WORKLOADS))
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--dump-cta", type=int, default=None, help="also list every event of this CTA, in time order")
    args = ap.parse_args()
    res = run(args.workload, args.launches, args.dump_cta)
    lines = res.pop("events", None)
    print(json.dumps(res))
    if lines:
        print("\n".join(lines))


if __name__ == "__main__":
    main()
