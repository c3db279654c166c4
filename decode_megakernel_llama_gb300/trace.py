"""Per-instruction trace of the megakernel (mk_set_trace / mk_read_trace).

Each record is {sm, op, wait_start_ns, start_ns, end_ns}: an instruction
waited on its dependency counter from wait_start to start and computed (and
consumed its weight pages) from start to end. This module turns a step's
records into per-op and per-SM time shares (wait = pipeline bubble, compute
= time inside instructions, idle = time an SM had no instruction) and into a
Chrome / Perfetto trace file.
"""
from __future__ import annotations

import json

import numpy as np

OP_NAMES = {1: "qkv", 2: "attn", 3: "oproj", 4: "gateup", 5: "down", 6: "lmhead"}


def summarize(rec: np.ndarray) -> dict:
    rec = np.asarray(rec, dtype=np.int64)
    if len(rec) == 0:
        return {}
    t0 = int(rec[:, 2].min())
    t1 = int(rec[:, 4].max())
    span = max(1, t1 - t0)
    out = {"span_us": span / 1e3, "n_instr": int(len(rec)), "ops": {}}
    for op, name in OP_NAMES.items():
        r = rec[rec[:, 1] == op]
        if len(r) == 0:
            continue
        wait = (r[:, 3] - r[:, 2]).sum()
        busy = (r[:, 4] - r[:, 3]).sum()
        out["ops"][name] = {"count": int(len(r)), "wait_us": wait / 1e3, "busy_us": busy / 1e3,
                            "mean_busy_us": busy / 1e3 / len(r)}
    sms = np.unique(rec[:, 0])
    waits, busys = [], []
    for s in sms:
        r = rec[rec[:, 0] == s]
        waits.append((r[:, 3] - r[:, 2]).sum())
        busys.append((r[:, 4] - r[:, 3]).sum())
    n = len(sms)
    out["sm_wait_frac"] = float(np.sum(waits) / (n * span))
    out["sm_busy_frac"] = float(np.sum(busys) / (n * span))
    out["sm_idle_frac"] = 1.0 - out["sm_wait_frac"] - out["sm_busy_frac"]
    return out


def to_chrome(rec: np.ndarray, path: str) -> None:
    rec = np.asarray(rec, dtype=np.int64)
    t0 = int(rec[:, 2].min()) if len(rec) else 0
    ev = []
    for sm, op, tw, ts, te in rec.tolist():
        name = OP_NAMES.get(op, str(op))
        if ts > tw:
            ev.append({"name": "wait", "ph": "X", "pid": 0, "tid": sm, "ts": (tw - t0) / 1e3,
                       "dur": (ts - tw) / 1e3, "cat": name})
        ev.append({"name": name, "ph": "X", "pid": 0, "tid": sm, "ts": (ts - t0) / 1e3,
                   "dur": (te - ts) / 1e3})
    with open(path, "w") as f:
        json.dump({"traceEvents": ev}, f)
