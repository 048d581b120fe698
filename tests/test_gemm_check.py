"""The comparison helpers themselves (no GPU): the output-grid rounding that
brackets the fused epilogue's allowed results."""
import numpy as np
import torch

from gemm_check import grid_round


def test_grid_points_are_fixed_points():
    rng = np.random.default_rng(0)
    bf = torch.from_numpy(rng.standard_normal(20000).astype(np.float32)).to(torch.bfloat16).double().numpy()
    h = (rng.standard_normal(20000) * np.logspace(-8, 4, 20000)).astype(np.float16).astype(np.float64)
    f = rng.standard_normal(20000).astype(np.float32).astype(np.float64)
    for vals, out in ((bf, "bf16"), (h, "f16"), (f, "f32")):
        assert np.array_equal(grid_round(vals, out, False), vals)
        assert np.array_equal(grid_round(vals, out, True), vals)


def test_between_neighbours_brackets_to_them():
    # bf16 neighbours of 1: 1 and 1 + 2^-7; f16 subnormal spacing 2^-24
    assert grid_round(np.array([1.003]), "bf16", False)[0] == 1.0
    assert grid_round(np.array([1.003]), "bf16", True)[0] == 1.0 + 2 ** -7
    assert grid_round(np.array([-1.003]), "bf16", False)[0] == -(1.0 + 2 ** -7)
    assert grid_round(np.array([1.5 * 2 ** -24]), "f16", False)[0] == 2 ** -24
    assert grid_round(np.array([1.5 * 2 ** -24]), "f16", True)[0] == 2 ** -23
    # the library's own round-to-nearest always lands inside the bracket
    x = np.random.default_rng(1).standard_normal(5000) * 100
    r = x.astype(np.float16).astype(np.float64)
    assert np.all(grid_round(x, "f16", False) <= r) and np.all(r <= grid_round(x, "f16", True))
