"""Per-instruction trace of the megakernel (mk_set_trace / mk_read_trace).

Each record is {sm, op, start - tile_wait, start, phase0, phase1, phase2,
end} in ns: an instruction ran from start to end, and thread 0 spent
tile_wait of that time waiting for weight / KV tiles to land in shared
memory. For a GEMV instruction phase0 ends its prologue
(input loaded and normalised), phase1 its tiles, phase2 its epilogue (the
rest is the release of its counters); for an attention instruction phase0
is the dependency met, phase1 q/k/v loaded, phase2 tiles done. This module
turns a step's records into per-op and per-SM time shares (wait = pipeline
bubble, busy = time inside instructions, idle = no instruction) and into a
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
    t0 = int(rec[:, 3].min())
    t1 = int(rec[:, 7].max())
    span = max(1, t1 - t0)
    out = {"span_us": span / 1e3, "n_instr": int(len(rec)), "ops": {}}
    for op, name in OP_NAMES.items():
        r = rec[rec[:, 1] == op]
        if len(r) == 0:
            continue
        wait = (r[:, 3] - r[:, 2]).sum()   # time spent waiting for tiles
        busy = (r[:, 7] - r[:, 3]).sum()
        ph = [float((r[:, 4] - r[:, 3]).mean()) / 1e3, float((r[:, 5] - r[:, 4]).mean()) / 1e3,
              float((r[:, 6] - r[:, 5]).mean()) / 1e3, float((r[:, 7] - r[:, 6]).mean()) / 1e3]
        out["ops"][name] = {"count": int(len(r)), "tile_wait_us": wait / 1e3, "busy_us": busy / 1e3,
                            "mean_busy_us": busy / 1e3 / len(r), "mean_phases_us": ph}
    sms = np.unique(rec[:, 0])
    waits, busys = [], []
    for s in sms:
        r = rec[rec[:, 0] == s]
        waits.append((r[:, 3] - r[:, 2]).sum())
        busys.append((r[:, 7] - r[:, 3]).sum())
    n = len(sms)
    out["sm_tile_wait_frac"] = float(np.sum(waits) / (n * span))
    out["sm_busy_frac"] = float(np.sum(busys) / (n * span))
    out["sm_idle_frac"] = 1.0 - out["sm_busy_frac"]
    return out


def to_chrome(rec: np.ndarray, path: str) -> None:
    rec = np.asarray(rec, dtype=np.int64)
    t0 = int(rec[:, 3].min()) if len(rec) else 0
    ev = []
    for sm, op, tw, ts, p0, p1, p2, te in rec.tolist():
        name = OP_NAMES.get(op, str(op))
        ev.append({"name": name, "ph": "X", "pid": 0, "tid": sm, "ts": (ts - t0) / 1e3,
                   "dur": (te - ts) / 1e3,
                   "args": {"tile_wait_us": (ts - tw) / 1e3, "phase0_us": (p0 - ts) / 1e3,
                            "phase1_us": (p1 - p0) / 1e3, "phase2_us": (p2 - p1) / 1e3}})
    with open(path, "w") as f:
        json.dump({"traceEvents": ev}, f)
