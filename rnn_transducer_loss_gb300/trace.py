"""Task trace of the persistent kernel (see rnnt_set_trace in include/rnnt_gb300.h).

``traced(fn)`` runs ``fn()`` with tracing on and returns the decoded records;
``summary(records)`` condenses them into the phase timeline: when the row
chunks, DP tasks and gradient chunks started and ended, how long each kind
ran per task, and how long the busiest SM was occupied.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _native as N

KINDS = ("row", "dp", "grad")


def traced(fn, max_tasks: int = 1 << 16, device="cuda"):
    buf = torch.full((max_tasks, 4), -1, dtype=torch.int32, device=device)
    rc = N.rnnt_set_trace(buf.data_ptr(), buf.numel() * 4)
    if rc != N.RNNT_OK:
        raise N.RNNTError(rc, "rnnt_set_trace")
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        N.rnnt_set_trace(None, 0)
    rec = buf.cpu().numpy()
    rec = rec[rec[:, 0] >= 0]
    return {"kind": rec[:, 0] & 3, "sample": rec[:, 0] >> 2, "sm": rec[:, 1],
            "start_us": rec[:, 2] / 1e3, "end_us": rec[:, 3] / 1e3}


def summary(r) -> dict:
    out = {}
    if len(r["kind"]) == 0:
        return {"tasks": 0}
    out["tasks"] = int(len(r["kind"]))
    out["span_us"] = float(r["end_us"].max() - min(0.0, r["start_us"].min()))
    for k, name in enumerate(KINDS):
        m = r["kind"] == k
        if not m.any():
            continue
        d = r["end_us"][m] - r["start_us"][m]
        out[name] = {"n": int(m.sum()), "first_start_us": float(r["start_us"][m].min()),
                     "last_end_us": float(r["end_us"][m].max()),
                     "mean_us": float(d.mean()), "max_us": float(d.max()),
                     "sum_us": float(d.sum())}
    dp = r["kind"] == 1
    if dp.any():
        out["dp_by_sample_us"] = {int(s): [float(a), float(b)] for s, a, b in
                                  zip(r["sample"][dp], r["start_us"][dp], r["end_us"][dp])}
    # Per sample: when its last row chunk ended, its DP ran, and its gradient
    # chunks started and ended (the critical path of the persistent kernel).
    per = {}
    for b in np.unique(r["sample"]):
        m = r["sample"] == b
        ent = {}
        for k, name in enumerate(KINDS):
            mk = m & (r["kind"] == k)
            if mk.any():
                ent[name] = [round(float(r["start_us"][mk].min()), 1),
                             round(float(r["end_us"][mk].max()), 1)]
        per[int(b)] = ent
    out["per_sample_us"] = per
    busy = {}
    for sm, a, b in zip(r["sm"], r["start_us"], r["end_us"]):
        busy[int(sm)] = busy.get(int(sm), 0.0) + float(b - a)
    v = np.array(list(busy.values()))
    out["sm_busy_us"] = {"min": float(v.min()), "mean": float(v.mean()), "max": float(v.max())}
    return out
