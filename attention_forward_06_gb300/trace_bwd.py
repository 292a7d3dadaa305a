"""Timeline of the backward kernels from their traced build (libattn_bwd_trace.so).

    python -m attention_forward_06_gb300.trace_bwd --workload train [--launches 4]

runs one forward of the workload (default library), then the backward through
the traced library (the same gradients as the default build, bit for bit),
reads the events of the last backward (include/attn_bwd_trace.h) and prints,
for each of the dK/dV and dQ kernels, where its time goes (medians over CTAs and
steps):

    span_us          first CTA start to last CTA end (the kernel's own extent)
    start_us         a CTA's start to its first S-type products
    step_us          interval between consecutive accumulating products inside an item
    item_cost_us     the extra time between an item's last accumulating product and the
                     next item's first, beyond one step (its epilogue, the next item's
                     tiles, the pipeline refilling)
    item_share       the CTAs' summed item costs over their summed time from start to end
    epilogue_us      accumulators complete to rows stored (compute warpgroup 0)
    compute_us       a step's S-type products ready to its P and dS handed over
    tail_us          spread of the CTAs' end times
    items_per_cta    work items a CTA processed

The recording adds a global store and a timer read per event, so the figures
run somewhat slower than the default build's.
"""
from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np
import torch

from . import _lib, ops
from .inputs import WORKLOADS, draw_workload

REC = np.dtype([("t", "<u8"), ("code", "<u4"), ("arg", "<u4")])
DKDV, DQ = 0, 1
PRODUCER, ISSUER, COMPUTE0, COMPUTE1 = range(4)
KERNEL_NAMES = ["dkdv", "dq"]


def read(lib) -> tuple[np.ndarray, np.ndarray]:
    """(counts [kernels, ctas, roles], records [kernels, ctas, roles, events]) of the launches since the last
    read."""
    dims = [ctypes.c_int() for _ in range(4)]
    lib.attn_bwd_trace_read(None, 0, *[ctypes.byref(d) for d in dims])
    kernels, ctas, roles, evs = (d.value for d in dims)
    n_bytes = 4 * kernels * ctas * roles
    r_bytes = REC.itemsize * kernels * ctas * roles * evs
    buf = (ctypes.c_uint8 * (n_bytes + r_bytes))()
    st = lib.attn_bwd_trace_read(buf, n_bytes + r_bytes, None, None, None, None)
    if st != 0:
        raise RuntimeError(f"attn_bwd_trace_read failed with status {st}")
    raw = np.frombuffer(buf, dtype=np.uint8)
    counts = raw[:n_bytes].view("<u4").reshape(kernels, ctas, roles).copy()
    recs = raw[n_bytes:].view(REC).reshape(kernels, ctas, roles, evs).copy()
    return counts, recs


def events(counts, recs, kernel, cta, role, code=None):
    """Kept events of one role of one CTA of one kernel (optionally of one code), in order."""
    n = min(int(counts[kernel, cta, role]), recs.shape[3])
    e = recs[kernel, cta, role, :n]
    return e if code is None else e[e["code"] == code]


def item_first(kernel: int, arg: int) -> bool:
    """Whether an accumulating-product event (code 11) is its item's first step."""
    return arg == 0 if kernel == DKDV else (arg & 1) == 0


def summarize(counts: np.ndarray, recs: np.ndarray, kernel: int) -> dict:
    """The figures listed in the module docstring, for one kernel."""
    ctas = [c for c in range(counts.shape[1]) if counts[kernel, c, PRODUCER] > 0]
    if not ctas:
        raise ValueError("no CTA recorded any event")
    starts, ends, first_s, steps, bounds, items, epi, comp, busy = [], [], [], [], [], [], [], [], []
    for c in ctas:
        t_start = int(events(counts, recs, kernel, c, PRODUCER, 0)["t"][0])
        done = events(counts, recs, kernel, c, ISSUER, 13)
        iss = events(counts, recs, kernel, c, ISSUER)
        starts.append(t_start)
        if len(done):
            ends.append(int(done["t"][-1]))
            busy.append(int(done["t"][-1]) - t_start)
        heads = iss[iss["code"] == 10]
        items.append(len(heads))
        if len(heads):
            first_s.append(int(heads["t"][0]) - t_start)
        acc = iss[iss["code"] == 11]
        for a, b in zip(acc[:-1], acc[1:]):
            (bounds if item_first(kernel, int(b["arg"])) else steps).append(int(b["t"]) - int(a["t"]))
        for role in (COMPUTE0, COMPUTE1):
            ev = events(counts, recs, kernel, c, role)
            ready = ev[ev["code"] == 20]["t"].astype(np.int64)
            hand = ev[ev["code"] == 21]["t"].astype(np.int64)
            n = min(len(ready), len(hand))
            comp.extend((hand[:n] - ready[:n]).tolist())
            if role == COMPUTE0:
                e0 = ev[ev["code"] == 23]["t"].astype(np.int64)
                e1 = ev[ev["code"] == 24]["t"].astype(np.int64)
                n = min(len(e0), len(e1))
                epi.extend((e1[:n] - e0[:n]).tolist())
    step = float(np.median(steps)) if steps else float("nan")
    item_cost = float(np.median(bounds)) - step if bounds else float("nan")
    extra = float(np.sum(np.maximum(np.array(bounds, dtype=np.float64) - step, 0.0))) if bounds else 0.0
    t0 = min(starts)
    return {
        "ctas": len(ctas),
        "span_us": (max(ends) - t0) / 1e3 if ends else float("nan"),
        "start_us": float(np.median(first_s)) / 1e3 if first_s else float("nan"),
        "step_us": step / 1e3,
        "steps": len(steps),
        "item_cost_us": item_cost / 1e3,
        "item_boundaries": len(bounds),
        "item_share": extra / float(np.sum(busy)) if busy else float("nan"),
        "epilogue_us": float(np.median(epi)) / 1e3 if epi else float("nan"),
        "compute_us": float(np.median(comp)) / 1e3 if comp else float("nan"),
        "tail_us": (max(ends) - min(ends)) / 1e3 if ends else float("nan"),
        "items_per_cta": float(np.mean(items)),
    }


def run(workload: str, launches: int = 4) -> dict:
    w = WORKLOADS[workload]
    lib = _lib.load("attn_bwd_trace", build_if_missing=True)
    dev = torch.device("cuda", 0)
    q, k, v = [t.to(dev) for t in draw_workload(w)]
    o, lse = ops.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    # the upstream gradient the benchmark's backward leg uses
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(w.seed + 5000)).to(torch.bfloat16).to(dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(ops.bwd_workspace_size(w.B, w.Hq, w.Sq), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(launches):
        flush.zero_()  # inputs come from HBM, as in the benchmark
        read(lib)  # keep only the last backward
        st = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.causal,
                          ctypes.c_float(w.scale), ws.data_ptr(), ws.numel(), stream)
        if st != 0:
            raise RuntimeError(f"attn_bwd failed with status {st}")
    counts, recs = read(lib)
    return {"workload": w.label(), **{KERNEL_NAMES[kk]: summarize(counts, recs, kk) for kk in (DKDV, DQ)}}


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="train", choices=sorted(WORKLOADS))
    ap.add_argument("--launches", type=int, default=4)
    args = ap.parse_args()
    print(json.dumps(run(args.workload, args.launches)))


if __name__ == "__main__":
    main()
