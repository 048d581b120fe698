"""Timeline trace of the tensor-core kernel.

With the options "trace_addr" / "trace_records" set (include/gemm.h,
gemm_trace_record_t), every role of the persistent kernel writes one record
per work unit -- the TMA producer's loads, the MMA issuer's accumulation, each
epilogue warp's drain of the accumulator -- plus one per CTA for its whole
life, each a %globaltimer span with the SM and CTA it ran on ("Learn CuTeDSL"
section 7: time stamps written by the kernel to a global buffer, turned into a
timeline on the host).  ``capture`` runs a function under tracing and returns
the records; ``chrome_trace`` lays them out for a Chrome-trace / Perfetto
viewer (one row per SM and role).
"""
from __future__ import annotations

import numpy as np

RECORD = np.dtype([("t_begin_ns", "<u8"), ("t_end_ns", "<u8"), ("unit", "<i4"), ("role", "<i2"), ("sm", "<i2"),
                   ("cta", "<i4"), ("sub", "<i4")])
ROLES = {1: "TMA loads", 2: "MMA", 3: "epilogue", 4: "CTA", 5: "set-up", 6: "epilogue detail"}
HEADER_BYTES = 32


def capture(fn, capacity: int = 1 << 16, device=None):
    """Run ``fn()`` (which enqueues library calls on the current stream) with
    tracing on, synchronise, and return (records, count): the records written
    as a structured array (at most ``capacity`` slots read; reserved slots a
    kernel thread did not fill, role 0, are skipped) and how many record
    slots the kernels reserved (at least the records written)."""
    import torch

    from . import GEMM_OK, GemmError, gemm_last_error, gemm_set_option

    assert RECORD.itemsize == 32
    buf = torch.zeros(HEADER_BYTES + RECORD.itemsize * capacity, dtype=torch.uint8,
                      device=device if device is not None else "cuda")
    for key, val in (("trace_records", capacity), ("trace_addr", buf.data_ptr())):
        if gemm_set_option(key, val) != GEMM_OK:
            raise GemmError(1, gemm_last_error())
    try:
        fn()
        torch.cuda.synchronize(buf.device)
    finally:
        gemm_set_option("trace_addr", 0)
        gemm_set_option("trace_records", 0)
    host = buf.cpu().numpy()
    count = int(host[:4].view(np.uint32)[0])
    n = min(count, capacity)
    recs = host[HEADER_BYTES:HEADER_BYTES + n * RECORD.itemsize].view(RECORD).copy()
    return recs[recs["role"] != 0], count


def chrome_trace(records) -> dict:
    """Chrome-trace JSON (complete events, microseconds from the first
    stamp): process = SM, thread = role (epilogue warps by lane quarter)."""
    if len(records) == 0:
        return {"traceEvents": []}
    t0 = int(records["t_begin_ns"].min())
    events = []
    for r in records:
        role = int(r["role"])
        name = ROLES.get(role, f"role {role}")
        tid = role * 10 + (int(r["sub"]) if role in (3, 5, 6) else 0)
        if role == 3 and int(r["sub"]) >= 4:
            name = "epilogue (to peer)"
        events.append({"name": name if role == 4 else f"{name} u{int(r['unit'])}", "ph": "X", "pid": int(r["sm"]),
                       "tid": tid, "ts": (int(r["t_begin_ns"]) - t0) / 1e3,
                       "dur": max(int(r["t_end_ns"]) - int(r["t_begin_ns"]), 0) / 1e3,
                       "args": {"unit": int(r["unit"]), "cta": int(r["cta"]), "sub": int(r["sub"])}})
    return {"traceEvents": events, "displayTimeUnit": "ns"}


def summary(records) -> dict:
    """Span of the traced launch(es) and per-role busy time, in microseconds:
    first CTA start to last CTA end, the mean CTA life, and per role the mean
    span per unit."""
    out = {}
    cta = records[records["role"] == 4]
    if len(cta):
        out["launch_us"] = (int(cta["t_end_ns"].max()) - int(cta["t_begin_ns"].min())) / 1e3
        out["cta_life_us_mean"] = float(np.mean(cta["t_end_ns"].astype(np.int64) - cta["t_begin_ns"].astype(np.int64))) / 1e3
    setup = records[(records["role"] == 5) & (records["sub"] == 0)]
    if len(setup):
        out["setup_us_mean"] = float(np.mean(setup["t_end_ns"].astype(np.int64) - setup["t_begin_ns"].astype(np.int64))) / 1e3
    for role, name in ((1, "loads"), (2, "mma"), (3, "epilogue")):
        sel = records[records["role"] == role]
        if len(sel):
            d = sel["t_end_ns"].astype(np.int64) - sel["t_begin_ns"].astype(np.int64)
            out[f"{name}_us_per_unit"] = float(np.mean(d)) / 1e3
    return out
