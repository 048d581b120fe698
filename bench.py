#!/usr/bin/env python3
"""Throughput benchmark of the GEMM library on GB300.

One step = one C = A.B through the C ABI (gemm_run) on the headline workload,
a BF16-input GEMM with M = N = K = 8192 (N(0,1) operands rounded to BF16, seed
3, FP32 accumulation and output) on the persistent tcgen05 path.  In the same
run, each of the other published workloads (FP32 SIMT and TF32 at 256^3 to
4096^3, the ragged BF16 shapes) is timed and checked against the oracle on
sampled rows; their compact records end the JSON line ("configs").  A
"sustained" leg repeats the headline back to back for over a second, against
the sustained peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Multi-GPU (torchrun): the GEMM is sharded by
rows -- each rank computes an 8192-row slab of a (ranks x 8192) x 8192 x 8192
product against its own copy of B, broadcast from rank 0 once before timing;
nothing crosses ranks inside the timed region (weak scaling); value = all
ranks' flops / the slowest rank's time.  --impl reference times the
fp64 oracle on the host cores on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s at 4096³/8192³ (FP32, TF32, BF16) and % of GB300 dense peak"
UNIT = "TFLOP/s"
L2_BYTES = 129e6
NOMINAL_DENSE_TFLOPS = {"bf16": 2250.0, "tf32": 1100.0, "fp8": 4500.0}   # GB300 per-GPU dense, nominal
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
FP32_LANES_PER_SM = 128
# bench keys of the published workloads (tiled_tensor_core_gemm_gb300/inputs.py)
WORKLOAD_KEYS = ("bf16_8192", "tf32_4096", "fp32_4096", "fp32_1024", "tf32_1024", "fp32_256",
                 "bf16_1000", "bf16_4097x4095x4099", "bf16_16384x1024x4096", "bf16_128x8192x8192",
                 "fp16_4096", "fp16_8192", "e4m3_4096", "e4m3_8192", "e5m2_8192")


# fused epilogues timed beside the plain GEMM (gemm_run_ex): bias + GELU with a
# BF16 C, and a residual add (beta = 1, the old BF16 C read back) with a BF16 C
FUSED_EPILOGUES = {"bias_gelu_bf16out": {"act": "gelu", "out": "bf16", "bias": True},
                   "residual_bf16out": {"beta": 1.0, "out": "bf16"}}


def workload_by_key(key):
    from tiled_tensor_core_gemm_gb300 import inputs as I
    table = {"bf16_8192": I.C4_BF16_8192, "tf32_4096": I.C3_TF32_4096, "fp32_4096": I.C3_FP32_4096,
             "fp32_1024": I.C2_FP32_1024, "tf32_1024": I.C2_TF32_1024, "fp32_256": I.C1_FP32_256,
             "bf16_1000": I.C5_BF16_RAGGED[0], "bf16_4097x4095x4099": I.C5_BF16_RAGGED[1],
             "bf16_16384x1024x4096": I.C5_BF16_RAGGED[2], "bf16_128x8192x8192": I.C5_BF16_RAGGED[3],
             "fp16_4096": I.FP16_4096, "fp16_8192": I.FP16_8192, "e4m3_4096": I.E4M3_4096,
             "e4m3_8192": I.E4M3_8192, "e5m2_8192": I.E5M2_8192}
    return table[key]


SHAPE_DTYPES = ("fp32", "tf32", "bf16", "fp16", "e4m3", "e5m2")


def shape_workload(spec: str, dtype: str):
    """A workload of any shape "MxNxK" (sizes >= 1) in one of the library's
    input types, operands U[-1,1] drawn from seed 4 like the ragged published
    shapes, for timing planner choices through the same path as the rest."""
    from tiled_tensor_core_gemm_gb300.inputs import Workload
    parts = spec.lower().split("x")
    if len(parts) != 3 or not all(p.isdigit() and int(p) >= 1 for p in parts):
        raise ValueError(f"--shape wants MxNxK with sizes >= 1, got {spec!r}")
    if dtype not in SHAPE_DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    M, N, K = (int(p) for p in parts)
    return Workload(f"{dtype} {M}x{N}x{K} U[-1,1] seed 4", M, N, K, dtype, "uniform", 4)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=tuple(WORKLOAD_KEYS), default="bf16_8192",
                    help="timed workload (default: the headline 8192^3 BF16 GEMM)")
    ap.add_argument("--shape", default=None, metavar="MxNxK",
                    help="time this shape instead of --workload (operands U[-1,1], seed 4; type from --dtype)")
    ap.add_argument("--dtype", choices=SHAPE_DTYPES, default="bf16", help="input type for --shape")
    ap.add_argument("--epilogue", choices=tuple(FUSED_EPILOGUES), default=None,
                    help="time the workload through gemm_run_ex with this fused epilogue")
    ap.add_argument("--grouped", choices=("equal_k", "skewed_k"), default=None,
                    help="time a 16-group BF16 grouped launch instead (equal K = 4096, or K log-uniform 512..8192)")
    ap.add_argument("--option", action="append", default=[], metavar="KEY=VALUE",
                    help="set a library option (gemm_set_option) for the whole run, e.g. tc_sched=2")
    ap.add_argument("--no-paths", action="store_true", help="skip the FP32/TF32 side paths")
    ap.add_argument("--trace", default=None, metavar="FILE",
                    help="after timing, trace one call of the workload in the kernel (per-unit, per-role time "
                         "stamps) and write it as Chrome-trace JSON to FILE; its summary joins the line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle time for cpu_baseline")
    return ap.parse_args()


# ---------------------------------------------------------------- helpers ---
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "sm_max_mhz")}, \
            "measured (MEASURED_PEAKS.json)"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback (no MEASURED_PEAKS.json)"


def source_digest(files) -> str:
    """Digest of a kernel's source files; profile figures taken from other sources are not reused."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tiled_tensor_core_gemm_gb300", "csrc")
    for name in files:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(key: str, plan: dict):
    """DRAM bytes per launch from a committed ncu summary (profiles/ncu_traffic.json),
    or None if the kernel's sources changed since that capture or this run's
    plan (tile, CTA group, K ranges, B staging, tail handling, schedule)
    differs from the one captured."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[key]
        if (d.get("source_digest") == source_digest(d["source_files"]) and "plan" in d
                and all(plan.get(k) == v for k, v in d["plan"].items())):
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling around a timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
            deadline = time.time() + 5
            while time.time() < deadline and os.path.getsize(self.file.name) == 0:
                time.sleep(0.02)
        except Exception:
            self.proc = None

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        with open(self.file.name) as f:
            text = f.read()
        os.unlink(self.file.name)
        rows = []
        for r in csv.reader(io.StringIO(text)):
            if len(r) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(r[2]), float(r[3]), float(r[4]), [x.strip() for x in r[5:10]]))
            except Exception:
                continue
        if not rows:
            return None
        inside = [x for x in rows if self.t0 - 1 <= x[0] <= self.t1 + 1] or rows
        reasons = set()
        names = ("active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for x in inside:
            for name, val in zip(names[1:], x[4][1:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": max(x[2] for x in inside),
                "power_w_max": max(x[3] for x in inside), "reasons": sorted(reasons), "samples": len(inside)}


def gpu_uuid(dev) -> str | None:
    try:
        import torch
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


# ------------------------------------------------------------ our timing ---
def make_device_operands(workload, device):
    from tiled_tensor_core_gemm_gb300.inputs import workload_operands
    A, B = workload_operands(workload)
    return A, B, A.to(device), B.to(device)


def time_gemm(tg, workload, steps, warmup, stream, device, dist=None, on_begin=None, on_end=None, epi=None):
    """Device-side timing with CUDA events on `stream`: one pair around all K
    steps, launched back to back as a user would (consecutive tensor-core
    launches overlap their set-up through programmatic dependent launch), so
    the average launch duration is that time / K; then a short pass with an
    event pair around each launch for the spread of single-launch times (an
    event between launches keeps them from overlapping, so these run a little
    longer).

    epi: None (gemm_run, FP32 C) or a fused epilogue for gemm_run_ex, as a dict
    with keys act, out, bias (bool), alpha, beta (seeded old C and bias)."""
    import torch
    _, _, A, B = make_device_operands(workload, device)
    if dist is not None:
        # row-sharded across ranks: this rank's slab of A is its own; B comes
        # from rank 0 once, into this rank's own buffer, before any timing
        from tiled_tensor_core_gemm_gb300.sharded import broadcast_b
        broadcast_b(B, 0)
        torch.cuda.synchronize(device)
    M, N, K = workload.M, workload.N, workload.K
    code = tg.DTYPES[workload.dtype]
    s = stream.cuda_stream
    if epi is None:
        C = torch.empty((M, N), dtype=torch.float32, device=device)
        plan = tg.gemm_plan(M, N, K, code, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N).as_dict()

        def run():
            rc = tg.gemm_run(M, N, K, code, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, s)
            if rc != tg.GEMM_OK:
                raise RuntimeError(tg.gemm_last_error())
    else:
        from tiled_tensor_core_gemm_gb300.inputs import make_epilogue_inputs
        c_old, bias = make_epilogue_inputs(M, N, epi["out"], workload.seed)
        C = c_old.to(device)
        bias_d = bias.to(device) if epi.get("bias") else None
        ep = tg.make_epilogue(epi.get("alpha", 1.0), epi.get("beta", 0.0),
                              bias_d.data_ptr() if bias_d is not None else 0, epi.get("act", "none"), epi["out"])
        plan = tg.gemm_plan(M, N, K, code, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N).as_dict()

        def run():
            rc = tg.gemm_run_ex(M, N, K, code, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N, ep, s)
            if rc != tg.GEMM_OK:
                raise RuntimeError(tg.gemm_last_error())

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run()
        stream.synchronize()
        st = tg.gemm_get_status(s)
        if st != tg.GEMM_OK:
            raise RuntimeError(f"warm-up status {st}: {tg.gemm_last_error()}")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        if on_begin:
            on_begin()
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        if on_end:
            on_end()
        if dist is not None:
            dist.barrier()
        total_ms = e0.elapsed_time(e1)
        st = tg.gemm_get_status(s)
        if st != tg.GEMM_OK:
            raise RuntimeError(f"timed-region status {st}: {tg.gemm_last_error()}")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(min(steps, 30))]
        for a, b in ev:
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    # the GEMM, plus the operand packs / B transpose before it and the split-K reduction after it
    launches = (1 + plan["pack_a"] + plan["pack_b"] + plan["b_kmajor"]
                + int(plan["tail_tiles"] > 0 and not plan.get("cluster_split"))
                if plan["path"] == 1 else 1)
    return {"total_ms": total_ms, "launch_ms_mean": total_ms / steps,
            "isolated_ms_mean": statistics.mean(launch_ms), "isolated_ms_median": statistics.median(launch_ms),
            "isolated_ms_min": min(launch_ms), "plan": plan, "launches_per_step": launches,
            "flops": 2.0 * M * N * K, "C": C}


class with_option:
    """Sets a library option for the duration of a block, then restores it."""

    def __init__(self, tg, key, value):
        self.tg, self.key, self.value = tg, key, value

    def __enter__(self):
        self.old = self.tg.gemm_get_option(self.key)
        if self.tg.gemm_set_option(self.key, self.value) != self.tg.GEMM_OK:
            raise RuntimeError(self.tg.gemm_last_error())

    def __exit__(self, *exc):
        self.tg.gemm_set_option(self.key, self.old)


def time_grouped(tg, workload, steps, warmup, stream, device, one_by_one=False, dist=None, on_begin=None,
                 on_end=None):
    """A grouped workload through gemm_run_grouped (one launch per step), or the
    same GEMMs through one gemm_run each; CUDA events around all steps."""
    import torch
    from tiled_tensor_core_gemm_gb300.inputs import grouped_operands
    pairs = [(A.to(device), B.to(device)) for A, B in grouped_operands(workload)]
    Cs = [torch.empty((A.shape[0], B.shape[1]), dtype=torch.float32, device=device) for A, B in pairs]
    code = tg.DTYPES[workload.dtype]
    s = stream.cuda_stream
    groups = [tg.GemmGroup(A.shape[0], B.shape[1], A.shape[1], A.data_ptr(), A.shape[1], B.data_ptr(), B.shape[1],
                           C.data_ptr(), C.shape[1], None) for (A, B), C in zip(pairs, Cs)]

    def run():
        if one_by_one:
            for (A, B), C in zip(pairs, Cs):
                rc = tg.gemm_run(A.shape[0], B.shape[1], A.shape[1], code, A.data_ptr(), A.shape[1], B.data_ptr(),
                                 B.shape[1], C.data_ptr(), C.shape[1], s)
                if rc != tg.GEMM_OK:
                    raise RuntimeError(tg.gemm_last_error())
        else:
            rc = tg.gemm_run_grouped(code, groups, None, s)
            if rc != tg.GEMM_OK:
                raise RuntimeError(tg.gemm_last_error())

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        if on_begin:
            on_begin()
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        if on_end:
            on_end()
        if dist is not None:
            dist.barrier()
    st = tg.gemm_get_status(s)
    if st != tg.GEMM_OK:
        raise RuntimeError(f"grouped status {st}: {tg.gemm_last_error()}")
    total = e0.elapsed_time(e1)
    ms = total / steps
    return {"ms": ms, "tflops": workload.flops / (ms * 1e-3) / 1e12, "total_ms": total, "launch_ms_mean": ms,
            "launch_ms_median": ms, "launch_ms_min": ms, "flops": workload.flops, "plan": None,
            "launches_per_step": len(pairs) if one_by_one else 1}


def time_e2e(tg, workload, steps, stream, device):
    """Same GEMM through gemm_run with the operands in pinned host memory: every
    step copies its A and B host->device, runs the GEMM, and copies C
    device->host.  Steps are pipelined over three streams with two device
    buffer sets -- step i's inputs copy in while step i-1 computes and step
    i-2's C copies out -- the way a serving loop overlaps transfers with
    compute; events order each buffer's reuse.  Time = first copy-in to last
    copy-out, divided by the steps."""
    import torch
    from tiled_tensor_core_gemm_gb300.inputs import workload_operands
    A_h, B_h = workload_operands(workload)
    A_h, B_h = A_h.pin_memory(), B_h.pin_memory()
    M, N, K = workload.M, workload.N, workload.K
    code = tg.DTYPES[workload.dtype]
    sets = []
    for _ in range(2):
        sets.append({"A": torch.empty_like(A_h, device=device), "B": torch.empty_like(B_h, device=device),
                     "C": torch.empty((M, N), dtype=torch.float32, device=device),
                     "C_h": torch.empty((M, N), dtype=torch.float32).pin_memory(),
                     "in": torch.cuda.Event(), "done": torch.cuda.Event(), "out": torch.cuda.Event(),
                     "used": False})
    h2d, comp, d2h = stream, torch.cuda.Stream(device), torch.cuda.Stream(device)

    def step(i):
        st = sets[i % 2]
        with torch.cuda.stream(h2d):
            if st["used"]:
                h2d.wait_event(st["done"])              # the GEMM that read this set has finished
            st["A"].copy_(A_h, non_blocking=True)
            st["B"].copy_(B_h, non_blocking=True)
            st["in"].record(h2d)
        comp.wait_event(st["in"])
        if st["used"]:
            comp.wait_event(st["out"])                  # this set's previous C has been copied out
        rc = tg.gemm_run(M, N, K, code, st["A"].data_ptr(), K, st["B"].data_ptr(), N, st["C"].data_ptr(), N,
                         comp.cuda_stream)
        if rc != tg.GEMM_OK:
            raise RuntimeError(tg.gemm_last_error())
        st["done"].record(comp)
        d2h.wait_event(st["done"])
        with torch.cuda.stream(d2h):
            st["C_h"].copy_(st["C"], non_blocking=True)
            st["out"].record(d2h)
        st["used"] = True

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d)
    comp.wait_event(e0)
    d2h.wait_event(e0)
    for i in range(steps):
        step(i)
    e1.record(d2h)                                      # after the last copy-out, which follows every step
    torch.cuda.synchronize()
    st = tg.gemm_get_status(comp.cuda_stream)
    if st != tg.GEMM_OK:
        raise RuntimeError(f"e2e status {st}: {tg.gemm_last_error()}")
    ms = e0.elapsed_time(e1) / steps
    h2d_b = A_h.numel() * A_h.element_size() + B_h.numel() * B_h.element_size()
    d2h_b = M * N * 4
    return ms, h2d_b, d2h_b


# ------------------------------------------------------ cpu_baseline leg ---
# The one place in the timed arm that runs the oracle: it times the oracle on a
# bounded sample of the workload, then checks sampled rows of the timed run's C
# against it.
def cpu_baseline_leg(workload, target_s, C_dev=None):
    """(cpu_baseline, parity): the oracle, as it stands, timed on a bounded
    sample of rows of the same GEMM; and, when C_dev (the timed run's C) is
    given, that C on sampled rows against the oracle's."""
    base = _time_oracle(workload, target_s)
    return base, (_parity_rows(workload, C_dev) if C_dev is not None else None)


def _time_oracle(workload, target_s):
    """The oracle, as it stands, on a bounded sample of rows of the same GEMM."""
    import oracle
    from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array, workload_operands
    A, B = workload_operands(workload)
    a, b = as_oracle_array(A), as_oracle_array(B)
    bf16, fp16 = workload.dtype == "bf16", workload.dtype == "fp16"
    fp8 = workload.dtype if workload.dtype in ("e4m3", "e5m2") else None
    threads = oracle.num_threads()
    rows = list(range(threads))
    t0 = time.perf_counter()
    oracle.gemm_rows(a, b, rows, bf16=bf16, fp16=fp16, fp8=fp8, with_scale=False)
    t_probe = time.perf_counter() - t0
    n = max(threads, int(threads * max(1.0, (target_s - t_probe) / max(t_probe, 1e-3))))
    n = min(n, workload.M)
    rows = list(range(n))
    t0 = time.perf_counter()
    oracle.gemm_rows(a, b, rows, bf16=bf16, fp16=fp16, fp8=fp8, with_scale=False)
    dt = time.perf_counter() - t0
    flops = 2.0 * n * workload.N * workload.K
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} of {workload.M} rows of C (each a full {workload.N}x{workload.K} row-panel product), "
                      f"fp64 C loops, {dt:.1f} s"}


TOL = {"fp32": 1e-5, "tf32": 2e-3, "bf16": 1e-5, "fp16": 1e-5, "e4m3": 1e-5, "e5m2": 1e-5}


def _parity_rows(workload, C_dev, nrows=32):
    """The timed run's C against the oracle on `nrows` rows spread over M (the
    first and last, the rest seeded): max |C - Cref| / (|A|.|B|) per entry."""
    import numpy as np
    import oracle
    from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array, workload_operands
    A, B = workload_operands(workload)
    rng = np.random.default_rng(workload.seed)
    rows = sorted({0, workload.M - 1, *(int(r) for r in rng.integers(0, workload.M, nrows - 2))})
    fp8 = workload.dtype if workload.dtype in ("e4m3", "e5m2") else None
    ref, D = oracle.gemm_rows(as_oracle_array(A), as_oracle_array(B), rows, bf16=workload.dtype == "bf16",
                              fp16=workload.dtype == "fp16", fp8=fp8, with_scale=True)
    got = C_dev[rows].double().cpu().numpy()
    finite = bool(np.all(np.isfinite(got)))
    zero = D == 0
    exact_zero = bool(np.all(got[zero] == ref[zero]))
    r = float(np.max(np.abs(got[~zero] - ref[~zero]) / D[~zero])) if np.any(~zero) else 0.0
    tol = TOL[workload.dtype]
    return {"rows": len(rows), "max_err_ratio": r, "tol": tol, "ok": finite and exact_zero and r <= tol,
            "what": "the timed run's C on sampled rows against the fp64 oracle, max |C - Cref| / (|A|.|B|)"}


def configs_parity(workload, C_dev, nrows=16):
    """A published workload's timed C against the oracle on sampled rows (part
    of the cpu_baseline leg: skipped with --no-cpu-baseline)."""
    return _parity_rows(workload, C_dev, nrows)


def slowest_rank_ms(total_ms: float, dist=None, device="cpu") -> float:
    """The timed region's length on the slowest rank (every rank gets the max)."""
    if dist is None:
        return total_ms
    import torch
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_tflops(world: int, flops_per_step: float, steps: int, max_total_ms: float) -> float:
    """Whole-job throughput of `world` independent replicas: all ranks' flops
    over the slowest rank's time."""
    return world * flops_per_step * steps / (max_total_ms * 1e-3) / 1e12


def roofline_tensor(flops, launch_ms, peak, peak_src, nominal, traffic):
    achieved = flops / (launch_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": UNIT,
            "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_src,
            "frac_of_nominal_dense": round(achieved / nominal, 4), "nominal_dense_peak": nominal}


ELEM_BYTES = {"fp32": 4, "tf32": 4, "bf16": 2, "fp16": 2, "e4m3": 1, "e5m2": 1}


def roofline_for_dtype(dtype, flops, launch_ms, peaks, peak_src, traffic):
    """Tensor roofline against the measured BF16 burst peak, scaled by the
    nominal dense ratio for TF32 (1100/2250) and FP8 (4500/2250)."""
    fam = {"tf32": "tf32", "e4m3": "fp8", "e5m2": "fp8"}.get(dtype, "bf16")
    ratio = NOMINAL_DENSE_TFLOPS[fam] / NOMINAL_DENSE_TFLOPS["bf16"]
    src = f"bf16_tflops burst, {peak_src}" if fam == "bf16" else f"bf16 burst x nominal {fam}/bf16 ratio, {peak_src}"
    return roofline_tensor(flops, launch_ms, peaks["bf16_tflops"] * ratio, src, NOMINAL_DENSE_TFLOPS[fam], traffic)


def roofline_alu(flops, launch_ms, sm_mhz, sms):
    """FP32 SIMT roofline: the FP32 FMA pipes of `sms` SMs (read from the
    device) at `sm_mhz`."""
    achieved = flops / (launch_ms * 1e-3) / 1e12
    peak = sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    return {"bound": "alu", "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": UNIT,
            "frac": round(achieved / peak, 4), "traffic": None,
            "peak_source": f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x {sm_mhz:.0f} MHz"}


def roofline_hbm(workload, launch_ms, peaks, peak_src, traffic):
    """HBM roofline of a GEMM too short and wide to be compute-bound: its
    compulsory bytes (A and B read once, C written once) per call."""
    in_bytes = (workload.M * workload.K + workload.K * workload.N) * ELEM_BYTES[workload.dtype]
    gbs = (in_bytes + workload.M * workload.N * 4) / (launch_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic, "peak_source": f"hbm_gbs, {peak_src}",
            "tensor_tflops": round(2.0 * workload.M * workload.N * workload.K / (launch_ms * 1e-3) / 1e12, 2)}


# The published workloads other than the headline, timed beside it; their
# compact records end the JSON line (key: the workload's id and shape).
CONFIG_WORKLOADS = (("c1_fp32_256", "fp32_256"), ("c2_fp32_1024", "fp32_1024"), ("c2_tf32_1024", "tf32_1024"),
                    ("c3_fp32_4096", "fp32_4096"), ("c3_tf32_4096", "tf32_4096"), ("c5_bf16_1000", "bf16_1000"),
                    ("c5_bf16_4097x4095x4099", "bf16_4097x4095x4099"),
                    ("c5_bf16_16384x1024x4096", "bf16_16384x1024x4096"),
                    ("c5_bf16_128x8192x8192", "bf16_128x8192x8192"))
# HBM-bound among them (B streams once past a few rows of A)
HBM_BOUND = {"bf16_128x8192x8192"}


def config_record(roof, parity):
    """Compact record of one published workload: throughput, the roofline it
    is judged against, and the timed run's C against the oracle on sampled rows."""
    rec = {"tflops": roof.get("tensor_tflops", roof["achieved"]), "bound": roof["bound"],
           "achieved": roof["achieved"], "peak": round(roof["peak"], 1), "unit": roof["unit"],
           "frac": round(roof["frac"], 3)}
    if parity is not None:
        rec["parity"] = float(f"{parity['max_err_ratio']:.2e}")
        rec["tol"] = parity["tol"]
        rec["ok"] = parity["ok"]
    return rec


def ordered_line(out):
    """The JSON line with the contract keys first and the compact per-config
    records last, so that the end of the line (the part of stdout a driver
    keeps) holds every published workload's figure."""
    last = ("paths", "sustained", "configs")
    d = {k: v for k, v in out.items() if k not in last}
    d.update({k: out[k] for k in last if k in out})
    return json.dumps(d, separators=(",", ":"))


def run_ours(args):
    import torch
    import tiled_tensor_core_gemm_gb300 as tg
    from tiled_tensor_core_gemm_gb300 import build as tgbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if rank == 0:
        tgbuild.build()
    if dist is not None:
        dist.barrier()
    tg.load_library()
    for kv in args.option:
        key, _, val = kv.partition("=")
        if tg.gemm_set_option(key, int(val)) != tg.GEMM_OK:
            raise SystemExit(f"--option {kv}: {tg.gemm_last_error()}")
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device)

    from tiled_tensor_core_gemm_gb300.inputs import GROUPED_BF16, GROUPED_BF16_SKEWK
    gw = {"equal_k": GROUPED_BF16, "skewed_k": GROUPED_BF16_SKEWK}.get(args.grouped)
    if gw is not None:
        w = gw
    elif args.shape:
        w = shape_workload(args.shape, args.dtype)
    else:
        w = workload_by_key(args.workload)
    wkey = (f"grouped_{args.grouped}" if gw is not None else
            f"{args.dtype}_{args.shape.lower()}" if args.shape else args.workload)
    headline = wkey == "bf16_8192" and not args.epilogue
    sampler = ClockSampler(gpu_uuid(device)) if rank == 0 else None
    if sampler:
        sampler.start()
    res = None
    try:
        hooks = dict(on_begin=sampler.mark_begin if sampler else None, on_end=sampler.mark_end if sampler else None)
        if gw is not None:
            res = time_grouped(tg, gw, args.steps, args.warmup, stream, device, dist=dist, **hooks)
        else:
            res = time_gemm(tg, w, args.steps, args.warmup, stream, device, dist, **hooks,
                            epi=FUSED_EPILOGUES[args.epilogue] if args.epilogue else None)
    finally:
        clocks = sampler.stop() if sampler else None

    total_ms = slowest_rank_ms(res["total_ms"], dist, device)
    ms_per_step = total_ms / args.steps
    value = replicas_tflops(world, res["flops"], args.steps, total_ms)

    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return

    if gw is not None:
        in_bytes = sum((m * gw.k_of(g) + gw.k_of(g) * gw.N) * ELEM_BYTES[gw.dtype] for g, m in enumerate(gw.Ms))
        shape = {"group_rows": list(gw.Ms), "group_k": [gw.k_of(g) for g in range(len(gw.Ms))], "N": gw.N}
    else:
        in_bytes = (w.M * w.K + w.K * w.N) * ELEM_BYTES[w.dtype]
        shape = {"M": w.M, "N": w.N, "K": w.K}
    desc = {"bf16_8192": "bf16-input GEMM M=N=K=8192, A,B ~ N(0,1) rounded to bf16 (seed 3), fp32 accumulate "
                         "and output, row-major, persistent tcgen05 path",
            "tf32_4096": "fp32 GEMM M=N=K=4096 read as TF32 by the tensor cores, A,B ~ N(0,1) (seed 2), fp32 "
                         "accumulate and output, row-major, persistent tcgen05 path",
            "fp32_4096": "fp32 GEMM M=N=K=4096, A,B ~ N(0,1) (seed 2), exact fp32 on the CUDA cores (SIMT)"}
    desc.setdefault(wkey, f"{w.name}, row-major, fp32 output" +
                    (", one gemm_run_grouped launch per step" if gw is not None else ""))
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    sm_mhz = (clocks or {}).get("sm_max_mhz") or peaks["sm_max_mhz"]

    def roofline_of(key, wl, r):
        """The roofline a workload is judged against: FP32 FMA pipes (SIMT),
        HBM (short and wide shapes), else the tensor cores of its input type."""
        if wl.dtype == "fp32":
            return roofline_alu(r["flops"], r["launch_ms_mean"], sm_mhz, sms)
        traffic = None if r["plan"] is None else profiled_traffic(key, r["plan"])
        if key in HBM_BOUND:
            return roofline_hbm(wl, r["launch_ms_mean"], peaks, peak_src, traffic)
        rl = roofline_for_dtype(wl.dtype, r["flops"], r["launch_ms_mean"], peaks, peak_src, traffic)
        if wl.dtype in ("bf16", "fp16"):
            rl["frac_of_sustained"] = round(rl["achieved"] / peaks["bf16_tflops_sustained"], 4)
        return rl

    roof = roofline_of(wkey + (f"_{args.epilogue}" if args.epilogue else ""), w, res)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": desc[wkey] + (f"; fused epilogue {FUSED_EPILOGUES[args.epilogue]} "
                                               "through gemm_run_ex" if args.epilogue else ""),
                   **shape, "parallelism": (f"rows x{world}: each rank the M-row slab above of a "
                                            f"{world * shape.get('M', 0)}-row GEMM, B broadcast once before timing"
                                            if world > 1 and gw is None else
                                            f"replicas x{world}" if world > 1 else "single"),
                   "options": args.option,
                   "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB of operands vs 129 MB L2); no flush",
                   "plan": res["plan"]},
        "roofline": roof,
        "kernel_ms": {"mean": round(res["launch_ms_mean"], 5),
                      "isolated_launches": {k: round(res[f"isolated_ms_{k}"], 5) for k in ("mean", "median", "min")}
                      if "isolated_ms_mean" in res else None},
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": clocks,
    }
    if args.trace and gw is None and rank == 0:
        from tiled_tensor_core_gemm_gb300 import trace as tt
        _, _, At, Bt = make_device_operands(w, device)
        Ct = torch.empty((w.M, w.N), dtype=torch.float32, device=device)

        def one_call():
            with torch.cuda.stream(stream):
                rc = tg.gemm_run(w.M, w.N, w.K, tg.DTYPES[w.dtype], At.data_ptr(), w.K, Bt.data_ptr(), w.N,
                                 Ct.data_ptr(), w.N, stream.cuda_stream)
                if rc != tg.GEMM_OK:
                    raise RuntimeError(tg.gemm_last_error())
        one_call()                                     # warm
        recs, count = tt.capture(one_call)
        with open(args.trace, "w") as f:
            json.dump(tt.chrome_trace(recs), f)
        out["trace"] = {"file": args.trace, "records": int(len(recs)), "slots": int(count),
                        **{k: round(v, 2) for k, v in tt.summary(recs).items()}}
        del At, Bt, Ct
    check = not args.no_cpu_baseline and world == 1
    if not args.no_paths and headline:
        n_side = max(3, min(args.steps, 100))
        side_warm = max(3, min(args.warmup, 10))
        # the other published workloads: compact records with parity on sampled rows
        configs = {}
        for cid, key in CONFIG_WORKLOADS:
            wl = workload_by_key(key)
            r = time_gemm(tg, wl, n_side, side_warm, stream, device)
            rl = roofline_of(key, wl, r)
            configs[cid] = config_record(rl, configs_parity(wl, r["C"]) if check else None)
            configs[cid]["plan"] = plan_tag(r["plan"])
            del r
        # more input types, fused epilogues and schedules on the pages' benchmark sizes
        paths = {}
        fused = {f"bf16_8192_{k}": v for k, v in FUSED_EPILOGUES.items()}
        extra = [(k, workload_by_key(k), None) for k in ("fp16_4096", "fp16_8192", "e4m3_4096", "e4m3_8192",
                                                        "e5m2_8192")]
        extra += [(k, workload_by_key("bf16_8192"), v) for k, v in fused.items()]
        for key, wl, epi in extra:
            r = time_gemm(tg, wl, n_side, side_warm, stream, device, epi=epi)
            rl = roofline_of(key, wl, r)
            paths[key] = {"tflops": rl["achieved"], "frac": round(rl["frac"], 3)}
        with with_option(tg, "tc_sched", 2):
            r = time_gemm(tg, w, n_side, side_warm, stream, device)
        rl = roofline_of("bf16_8192_dynamic_schedule", w, r)
        paths["bf16_8192_dynamic_schedule"] = {"tflops": rl["achieved"], "frac": round(rl["frac"], 3)}
        from tiled_tensor_core_gemm_gb300.inputs import GROUPED_BF16, GROUPED_BF16_SKEWK
        # 16-group workloads: one grouped launch (static / dynamic / automatic schedule), and as 16 calls
        for key, gwl, obo, sched in (("grouped_bf16_16", GROUPED_BF16, False, 1),
                                    ("grouped_bf16_16_dynamic_schedule", GROUPED_BF16, False, 2),
                                    ("grouped_bf16_16_one_by_one", GROUPED_BF16, True, 1),
                                    ("grouped_bf16_16_skewed_k_static_schedule", GROUPED_BF16_SKEWK, False, 1),
                                    ("grouped_bf16_16_skewed_k", GROUPED_BF16_SKEWK, False, 0)):
            with with_option(tg, "tc_sched", sched):
                r = time_grouped(tg, gwl, n_side, side_warm, stream, device, obo)
            rl = roofline_for_dtype("bf16", gwl.flops, r["ms"], peaks, peak_src, None)
            paths[key] = {"tflops": rl["achieved"], "frac": round(rl["frac"], 3)}
        out["paths"] = paths
        # the headline again, back to back for at least a second: the clock the
        # power cap settles at, against the sustained peak
        sus_steps = max(args.steps, int(1.2 / max(ms_per_step * 1e-3, 1e-6)) + 1)
        sus_sampler = ClockSampler(gpu_uuid(device))
        sus_sampler.start()
        try:
            r = time_gemm(tg, w, sus_steps, 3, stream, device, on_begin=sus_sampler.mark_begin,
                          on_end=sus_sampler.mark_end)
        finally:
            sus_clocks = sus_sampler.stop()
        sus_tf = r["flops"] / (r["launch_ms_mean"] * 1e-3) / 1e12
        out["sustained"] = {"tflops": round(sus_tf, 2), "steps": sus_steps, "seconds": round(r["total_ms"] / 1e3, 2),
                            "peak": peaks["bf16_tflops_sustained"],
                            "frac": round(sus_tf / peaks["bf16_tflops_sustained"], 4),
                            "frac_of_burst": round(sus_tf / peaks["bf16_tflops"], 4), "clocks": sus_clocks}
        del r
        out["configs"] = configs

    if not args.no_e2e and gw is None:
        ms, h2d, d2h = time_e2e(tg, w, max(3, min(args.steps, 50)), stream, device)
        out["e2e"] = {"value": round(world * 2.0 * w.M * w.N * w.K / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
                      "how": "pinned host A,B -> device, gemm_run, C -> pinned host each step, pipelined over "
                             "three streams; events from the first copy-in to the last copy-out"}
    if check and gw is None:
        out["cpu_baseline"], parity = cpu_baseline_leg(w, args.cpu_seconds, None if args.epilogue else res["C"])
        if parity is not None:
            out["parity"] = parity
            if "configs" in out:
                out["configs"] = {"c4_bf16_8192": config_record(roof, parity) | {"plan": plan_tag(res["plan"])},
                                  **out["configs"]}
    print(ordered_line(out), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def plan_tag(plan):
    """The plan in a few characters: CTA group x tile width, K ranges or
    column halves, B staging, packs and store path."""
    if plan is None:
        return None
    if plan["path"] == 0:
        return f"simt{plan['bm']}x{plan['bn']}" + (f"/k{plan['splits']}" if plan["splits"] > 1 else "")
    t = f"cg{plan['cta_group']}x{plan['bn']}"
    if plan["tail_tiles"]:
        t += f"/k{plan['splits']}" + ("" if plan["tail_tiles"] == plan["tiles"] else "tail")
        t += "dsm" if plan.get("cluster_split") else ""
        t += f"{plan['kb_split']}" if plan.get("kb_split") else ""
    if plan["half_tiles"]:
        t += "/halves"
    if plan["b_kmajor"]:
        t += "/bT"
    if plan["pack_a"] or plan["pack_b"]:
        t += "/pack" + ("A" if plan["pack_a"] else "") + ("B" if plan["pack_b"] else "")
    if not plan["tma_store"]:
        t += "/st"
    return t


# -------------------------------------------------------- reference arm ---
def run_reference(args):
    """The fp64 oracle on the host cores, each step a bounded sample of rows of
    the same 8192^3 BF16 GEMM."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from tiled_tensor_core_gemm_gb300.inputs import C4_BF16_8192 as w, as_oracle_array, workload_operands
    oracle.build()
    A, B = workload_operands(w)
    a, b = as_oracle_array(A), as_oracle_array(B)
    threads = oracle.num_threads()
    t0 = time.perf_counter()
    oracle.gemm_rows(a, b, list(range(threads)), bf16=True, with_scale=False)
    t_step = time.perf_counter() - t0
    budget = 150.0
    rows = threads
    if t_step * (args.steps + args.warmup) > budget:
        rows = max(1, int(threads * budget / (t_step * (args.steps + args.warmup))))
    sample = list(range(rows))
    for i in range(args.warmup):
        oracle.gemm_rows(a, b, [(r + i * rows) % w.M for r in sample], bf16=True, with_scale=False)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.gemm_rows(a, b, [(r + i * rows) % w.M for r in sample], bf16=True, with_scale=False)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / dt / 1e12
    used = min(rows, threads)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "bf16-input GEMM M=N=K=8192, A,B ~ N(0,1) rounded to bf16 (seed 3), "
                                  "fp32 accumulate and output, row-major; oracle on bounded row samples",
                      "M": w.M, "N": w.N, "K": w.K},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                            "sample": f"each step: {rows} rows of C of the 8192^3 GEMM (fp64 loops)"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps must be >= 1 and --warmup >= 0")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
