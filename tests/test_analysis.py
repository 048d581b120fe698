"""Pins for the closed-form models against the values the pages print (no GPU)."""
import os

import pytest

from tiled_tensor_core_gemm_gb300 import analysis

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_traffic_table_reproduces_printed_values():
    rows = _rows("traffic_n4096.txt")
    printed = {r[0]: (float(r[1]), float(r[2])) for r in rows if r[0] != "compulsory_MB"}
    ours = {name: (b, fpb) for name, b, fpb in analysis.traffic_table(4096)}
    assert set(printed) == set(ours)
    for name, (gb, fpb) in printed.items():
        b, f = ours[name]
        assert round(b / 1e9, 1) == gb, name
        assert round(f, 1) == fpb, name
    comp = [r for r in rows if r[0] == "compulsory_MB"][0]
    assert round(analysis.compulsory_read_bytes(4096, 4096, 4096, 4) / 1e6) == int(comp[1])


@pytest.mark.parametrize("T", [16, 32, 64, 128, 256])
def test_square_tile_intensity_is_T_over_4(T):
    assert analysis.block_tile_intensity(T, T) == T / 4
    n = 1024
    flops = analysis.gemm_flops(n, n, n)
    assert flops / analysis.block_tile_read_bytes(n, n, n, T, T) == pytest.approx(T / 4)


def test_bank_model_reproduces_printed_passes():
    printed = {r[0]: int(r[2]) for r in _rows("bank_passes.txt")}
    T, k = 16, 3

    def tid16(t):
        return t // T, t % T

    ours = {
        "store_sA_ty*T+tx": analysis.bank_passes(lambda t: tid16(t)[0] * T + tid16(t)[1]),
        "load_sA_ty*T+k": analysis.bank_passes(lambda t: tid16(t)[0] * T + k),
        "load_sB_k*T+tx": analysis.bank_passes(lambda t: k * T + tid16(t)[1]),
        "load_s_tx*32+k": analysis.bank_passes(lambda t: (t % 32) * 32 + k),
        "load_s_tx*33+k": analysis.bank_passes(lambda t: (t % 32) * 33 + k),
    }
    assert ours == printed


def test_flop_convention_and_8192_reading():
    for name, us, tf in _rows("tflops_8192.txt"):
        # durations are printed to the microsecond, so allow one TFLOP/s of rounding
        ours = analysis.tflops(analysis.gemm_flops(8192, 8192, 8192), float(us) * 1e-6)
        assert abs(ours - int(tf)) < 1.0, name
    # the page's "8096" label does not reproduce the printed throughput
    assert abs(analysis.tflops(analysis.gemm_flops(8096, 8096, 8096), 677e-6) - 1624) > 50


def test_fp32_peak_arithmetic():
    # 152 SMs x 128 FP32 lanes x 2 flop x 2070 MHz
    assert analysis.fp32_simt_peak_tflops(152, 2070.0) == pytest.approx(80.5478, rel=1e-4)
