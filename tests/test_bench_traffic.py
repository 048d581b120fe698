"""The DRAM traffic that bench.py puts in its roofline comes from committed
ncu captures (profiles/ncu_traffic.json).  A figure is only reported while
the kernel sources still hash to the captured digest and the run's plan is the
captured one; otherwise the roofline carries traffic null.  No GPU: plans come
from the library's planner for a 152-SM GB300."""
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
