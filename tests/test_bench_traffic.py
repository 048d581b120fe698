"""bench.py's host-side arithmetic, without a GPU.

The DRAM traffic in its roofline comes from committed ncu captures
(profiles/ncu_traffic.json).  A figure is only reported while the kernel
sources still hash to the captured digest and the run's plan is the captured
one; otherwise the roofline carries traffic null.  Plans come from the
library's planner for a 152-SM GB300.  Also: the --shape parser, and the
tensor and ALU roofline formulas on worked numbers."""
import json
import os

import pytest

import bench
import tiled_tensor_core_gemm_gb300 as tg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
SHAPES = {"bf16_8192": (8192, 8192, 8192, tg.GEMM_BF16), "bf16_8192_bias_gelu_bf16out": (8192, 8192, 8192, tg.GEMM_BF16),
          "bf16_8192_residual_bf16out": (8192, 8192, 8192, tg.GEMM_BF16),
          "tf32_4096": (4096, 4096, 4096, tg.GEMM_TF32), "e4m3_8192": (8192, 8192, 8192, tg.GEMM_E4M3),
          "bf16_128x8192x8192": (128, 8192, 8192, tg.GEMM_BF16)}


def _plan(M, N, K, dt):
    return tg.gemm_plan(M, N, K, dt, 0, K, 0, N, 0, N, 152).as_dict()


def test_every_capture_names_its_plan_and_sources():
    assert set(TABLE) == set(SHAPES)
    for key, d in TABLE.items():
        assert {"cta_group", "bn", "splits", "b_kmajor", "tail_tiles", "half_tiles", "sched"} <= set(d["plan"]), key
        assert d["dram_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_write"], key
        assert os.path.exists(os.path.join(ROOT, d["capture"])), key


@pytest.mark.parametrize("key", sorted(SHAPES))
def test_traffic_reported_only_for_the_captured_plan(key):
    d = TABLE[key]
    plan = _plan(*SHAPES[key])
    same = all(plan[k] == v for k, v in d["plan"].items())
    digest_ok = d["source_digest"] == bench.source_digest(d["source_files"])
    got = bench.profiled_traffic(key, plan)
    assert got == (float(d["dram_bytes_per_launch"]) if same and digest_ok else None)
    # any other tile width is a different kernel instance: no figure
    other = dict(plan, bn=128 if plan["bn"] == 256 else 256)
    assert bench.profiled_traffic(key, other) is None
    assert bench.profiled_traffic("no_such_workload", plan) is None


def test_headline_capture_matches_the_current_plan_and_sources():
    assert bench.profiled_traffic("bf16_8192", _plan(8192, 8192, 8192, tg.GEMM_BF16)) is not None


def test_shape_workload_parses_and_rejects():
    w = bench.shape_workload("128x8192X8192", "bf16")
    assert (w.M, w.N, w.K, w.dtype, w.dist, w.seed) == (128, 8192, 8192, "bf16", "uniform", 4)
    for bad in ("128x8192", "0x8x8", "ax8x8", "8x8x8x8", "-1x8x8"):
        with pytest.raises(ValueError):
            bench.shape_workload(bad, "bf16")
    with pytest.raises(ValueError):
        bench.shape_workload("8x8x8", "int8")


# ----------------------------------------------------- roofline arithmetic --
PEAKS = {"hbm_gbs": 6778.0, "bf16_tflops": 1905.1, "bf16_tflops_sustained": 1693.7, "sm_max_mhz": 2070.0}


def test_tensor_roofline_worked_headline():
    # 2 * 8192^3 flop in 0.6598 ms per launch is 1666.4 TFLOP/s, 0.8747 of the 1905.1 burst peak
    r = bench.roofline_for_dtype("bf16", 2 * 8192 ** 3, 0.6598, PEAKS, "measured", 1.37e9)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] == 1.37e9
    assert r["achieved"] == pytest.approx(1666.4, abs=0.1) and r["peak"] == 1905.1
    assert r["frac"] == pytest.approx(0.8747, abs=1e-4)
    assert r["frac_of_nominal_dense"] == pytest.approx(1666.4 / 2250, abs=1e-4)


@pytest.mark.parametrize("dtype,peak", [("fp16", 1905.1), ("tf32", 931.4), ("e4m3", 3810.2), ("e5m2", 3810.2)])
def test_tensor_peak_per_input_type(dtype, peak):
    # the measured BF16 burst peak scaled by the nominal dense ratio (TF32 1100/2250, FP8 4500/2250)
    r = bench.roofline_for_dtype(dtype, 1e12, 1.0, PEAKS, "measured", None)
    assert r["peak"] == pytest.approx(peak, abs=0.05)
    assert r["achieved"] == pytest.approx(1000.0) and r["frac"] == pytest.approx(1000.0 / peak, abs=1e-4)


def test_alu_roofline_worked_fp32():
    # 152 SMs x 128 FP32 lanes x 2 flop x 2070 MHz = 80.55 TFLOP/s; 4096^3 in 2.466 ms is 55.7 of it
    r = bench.roofline_alu(2 * 4096 ** 3, 2.466, 2070.0, 152)
    assert r["bound"] == "alu" and r["peak"] == pytest.approx(80.55, abs=0.01)
    assert r["achieved"] == pytest.approx(55.73, abs=0.01) and r["frac"] == pytest.approx(0.6919, abs=1e-4)


def test_cpu_baseline_leg_times_the_oracle_and_checks_sampled_rows():
    import torch
    import oracle
    from tiled_tensor_core_gemm_gb300.inputs import Workload, as_oracle_array, workload_operands
    w = Workload("bf16 96x80x64 U[-1,1] seed 4", 96, 80, 64, "bf16", "uniform", 4)
    A, B = workload_operands(w)
    good = torch.from_numpy(oracle.gemm(as_oracle_array(A), as_oracle_array(B), bf16=True).astype("float32"))
    base, parity = bench.cpu_baseline_leg(w, 0.05, good)
    assert base["kind"] == "oracle" and base["unit"] == "TFLOP/s" and base["value"] > 0 and base["cores"] >= 1
    assert parity["ok"] and parity["max_err_ratio"] <= 1e-7 and parity["rows"] >= 2
    bad = good.clone()
    bad[0, 5] += 1.0                   # row 0 is always sampled
    assert not bench.cpu_baseline_leg(w, 0.05, bad)[1]["ok"]
    nan = good.clone()
    nan[w.M - 1, 0] = float("nan")     # and so is the last row
    assert not bench.cpu_baseline_leg(w, 0.05, nan)[1]["ok"]
    assert bench.cpu_baseline_leg(w, 0.05, None)[1] is None


def test_hbm_roofline_worked_short_wide_shape():
    # 128 x 8192 x 8192 BF16: (128*8192 + 8192*8192) * 2 + 128*8192*4 bytes = 140.5 MB in 26.0 us is 5404 GB/s
    from tiled_tensor_core_gemm_gb300.inputs import C5_BF16_RAGGED
    r = bench.roofline_hbm(C5_BF16_RAGGED[3], 0.026, PEAKS, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6778.0
    assert r["achieved"] == pytest.approx(140.5e6 / 26.0e-6 / 1e9, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / 6778.0, abs=1e-4)
    assert r["tensor_tflops"] == pytest.approx(2 * 128 * 8192 * 8192 / 26.0e-6 / 1e12, abs=0.01)


def test_configs_record_ends_the_line_within_a_short_tail():
    """A line shaped like the headline run's, with every published workload:
    the per-config object comes last, so the last 2000 characters of stdout
    (all a driver may keep) hold it whole."""
    import json
    roof = bench.roofline_for_dtype("bf16", 2 * 8192 ** 3, 0.5763, PEAKS, "measured", 1373747080.0)
    parity = {"rows": 32, "max_err_ratio": 9.3e-7, "tol": 1e-5, "ok": True, "what": "x" * 80}
    plan = {"path": 1, "cta_group": 2, "bn": 256, "tail_tiles": 64, "tiles": 64, "splits": 2, "half_tiles": 0,
            "b_kmajor": 0, "pack_a": 1, "pack_b": 1, "tma_store": 0, "bm": 128}
    configs = {cid: bench.config_record(roof, parity) | {"plan": bench.plan_tag(plan)}
               for cid, _ in (("c4_bf16_8192", 0),) + bench.CONFIG_WORKLOADS}
    out = {"metric": bench.METRIC, "value": 1907.8, "config": {"workload": "w" * 300, "plan": plan},
           "configs": configs, "roofline": roof, "paths": {f"p{i}": {"tflops": 1.0, "frac": 0.5} for i in range(12)},
           "sustained": {"tflops": 1666.0, "clocks": {"sm_mhz": 1515.0, "reasons": ["sw_power_cap"]}},
           "cpu_baseline": {"value": 0.04, "sample": "s" * 120}, "e2e": {"value": 662.8}, "parity": parity}
    line = bench.ordered_line(out)
    d = json.loads(line)
    assert list(d)[-1] == "configs" and list(d)[:2] == ["metric", "value"]
    tail = line[-2000:]
    assert tail.index('"configs":') >= 0 and line.endswith("}}}")
    assert json.loads("{" + tail[tail.index('"configs":'):]) == {"configs": configs}
    assert bench.plan_tag(plan) == "cg2x256/k2/packAB/st"
