"""The benchmark's JSON line on a short run: every key of the output contract
is present and consistent (a regression guard for bench.py itself)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_headline_line_has_every_contract_key():
    d = _run("--steps", "3", "--warmup", "3", "--no-paths", "--cpu-seconds", "1")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert set(d["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert set(d["cpu_baseline"]) >= {"value", "unit", "cores", "kind", "sample"} and d["cpu_baseline"]["kind"] == "oracle"
    assert set(d["e2e"]) >= {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert d["e2e"]["h2d_bytes_per_step"] == 2 * 8192 * 8192 * 2 and d["e2e"]["d2h_bytes_per_step"] == 8192 * 8192 * 4
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert d["gpu_launches"] == 3 and d["config"]["workload"]
    assert d["parity"]["ok"] and d["parity"]["rows"] >= 8 and d["parity"]["max_err_ratio"] <= 1e-5


def test_grouped_line():
    d = _run("--grouped", "skewed_k", "--steps", "3", "--warmup", "3", "--no-paths")
    assert d["value"] > 0 and d["gpu_launches"] == 3 and len(d["config"]["group_k"]) == 16
