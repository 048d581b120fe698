"""The comparison helpers themselves (no GPU): the output-grid rounding that
brackets the fused epilogue's allowed results, and the acceptance gate of the
parity tests against simulated correct and wrong kernel outputs."""
import numpy as np
import pytest
import torch

import oracle
from gemm_check import TOL, epilogue_check, error_ratio, grid_round, grid_round_nearest
from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array, make_operands


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


# ------------------------------------------------------- the acceptance gate --
# error_ratio is the parity gate of every GPU test: r = max |C - Cref| / D,
# with D = |A|.|B|.  These checks hand it what correct kernels produce (FP32
# sums in another order, blocked as a tile loop would; narrow inputs with FP32
# accumulation) and what plausible kernel bugs produce, simulated on the CPU,
# and require that the first pass the bound and the second fail it.
M, N, K = 300, 260, 1000
OUT = {"bf16": torch.bfloat16, "f16": torch.float16}
P = {"bf16": 8, "f16": 11}      # significand bits of the output type


def _ref(dtype="fp32", seed=31):
    A, B = make_operands(M, N, K, dtype, "normal", seed)
    a, b = as_oracle_array(A), as_oracle_array(B)
    Cref, D = oracle.gemm(a, b, bf16=(dtype == "bf16"), with_scale=True)
    return A.float().numpy().astype(np.float64), B.float().numpy().astype(np.float64), Cref, D


def _blocked_fp32(A, B, bk=64):
    """FP32 accumulation over K in blocks of bk, the way a tiled kernel sums."""
    acc = np.zeros((A.shape[0], B.shape[1]), np.float32)
    for k0 in range(0, A.shape[1], bk):
        acc = acc + (A[:, k0:k0 + bk].astype(np.float32) @ B[k0:k0 + bk].astype(np.float32))
    return acc


def test_correct_fp32_accumulation_passes():
    A, B, Cref, D = _ref()
    for bk in (1, 16, 64, K):
        assert error_ratio(_blocked_fp32(A, B, bk), Cref, D) <= TOL["fp32"]


def test_bf16_inputs_with_fp32_accumulation_pass():
    A, B, Cref, D = _ref("bf16")
    assert error_ratio(_blocked_fp32(A, B, 64), Cref, D) <= TOL["bf16"]


def _bugs(A, B, C):
    tail = _blocked_fp32(A[:, :K - 16], B[:K - 16])                     # last 16 of K never loaded
    swapped = C.copy()
    swapped[[*range(0, 128), *range(128, 256)]] = C[[*range(128, 256), *range(0, 128)]]  # two tiles' rows swapped
    shifted = C.copy()
    shifted[:, 256:259] = C[:, 257:260]                                  # ragged last tile one column off
    stale = C.copy()
    stale[128:256, :128] += C[:128, :128]                                # accumulator not cleared between tiles
    split_twice = C + _blocked_fp32(A[:, :256], B[:256])                 # a K range added twice
    split_missing = C - _blocked_fp32(A[:, 512:768], B[512:768])         # a K range left out
    unwritten = C.copy()
    unwritten[-3:] = np.nan                                              # last rows never stored
    half = C.copy()
    half[:, 128:] = 0.0                                                  # one column half never stored
    return {"k_tail": tail, "tiles_swapped": swapped, "column_shift": shifted, "stale_accumulator": stale,
            "k_range_twice": split_twice, "k_range_missing": split_missing, "rows_unwritten": unwritten,
            "column_half_unwritten": half}


def test_plausible_kernel_bugs_fail():
    A, B, Cref, D = _ref()
    C = _blocked_fp32(A, B)
    passed = {name: r for name, bad in _bugs(A, B, C).items() if (r := error_ratio(bad, Cref, D)) <= TOL["fp32"]}
    assert not passed, passed


def test_transposed_operand_fails():
    rng = np.random.default_rng(32)
    A = rng.standard_normal((96, 96)).astype(np.float32)
    B = rng.standard_normal((96, 96)).astype(np.float32)
    Cref, D = oracle.gemm(A, B, with_scale=True)
    assert error_ratio(A.astype(np.float32) @ B.T, Cref, D) > TOL["fp32"]
    assert error_ratio(A @ B, Cref, D) <= TOL["fp32"]


def test_one_element_just_outside_the_bound_fails():
    A, B, Cref, D = _ref()
    C = Cref.copy()
    C[17, 23] += 1.01 * TOL["fp32"] * D[17, 23]
    assert TOL["fp32"] < error_ratio(C, Cref, D) < 1.02 * TOL["fp32"]
    C[17, 23] = Cref[17, 23] + 0.99 * TOL["fp32"] * D[17, 23]
    assert error_ratio(C, Cref, D) <= TOL["fp32"]


def test_non_finite_and_zero_scale_cells():
    Cref = np.array([[1.0, 0.0]])
    D = np.array([[2.0, 0.0]])
    assert error_ratio(np.array([[1.0, 0.0]]), Cref, D) == 0.0
    assert error_ratio(np.array([[np.inf, 0.0]]), Cref, D) == float("inf")
    assert error_ratio(np.array([[np.nan, 0.0]]), Cref, D) == float("inf")
    # D = 0 (a zero row of A or column of B) leaves no room: anything but the exact value fails
    assert error_ratio(np.array([[1.0, 1e-30]]), Cref, D) == float("inf")
    assert error_ratio(np.zeros((0, 4)), np.zeros((0, 4)), np.zeros((0, 4))) == 0.0


def _grid_steps_up(x, out, n):
    """The n-th grid point of the output type above a positive grid value x."""
    for _ in range(n):
        x = grid_round(np.array([x * (1 + 2.0 ** -(P[out] + 1))]), out, True)[0]
    return x


@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_epilogue_gate_takes_the_rounded_value_and_rejects_one_step_beyond(out):
    A, B, Cref, D = _ref()
    bias = torch.linspace(-1, 1, N, dtype=torch.float32)
    args = ("fp32", out, 0.5, 0.0, None, bias, "gelu")
    y = oracle.epilogue(Cref, 0.5, 0.0, None, out, bias.numpy(), "gelu")
    # a correct kernel: FP32 sums, the epilogue in FP32, cast by round-to-nearest
    v = torch.from_numpy(_blocked_fp32(A, B)) * 0.5 + bias
    v = torch.nn.functional.gelu(v)
    good = v.to(OUT[out]).double().numpy()
    worst, y2 = epilogue_check(good, Cref, D, *args)
    assert np.array_equal(y, y2) and worst <= 1.0
    # the same output with its largest element one grid step above the rounded value
    i, j = np.unravel_index(np.argmax(y), y.shape)
    bad = good.copy()
    bad[i, j] = _grid_steps_up(good[i, j], out, 1)
    assert epilogue_check(bad, Cref, D, *args)[0] > 1.0
    bad[i, j] = np.nan
    assert epilogue_check(bad, Cref, D, *args)[0] == float("inf")


def test_grid_round_nearest_matches_the_library_casts():
    """Round-to-nearest-even onto each output grid, against the library's own
    FP32 -> BF16 / FP16 and FP64 -> FP32 conversions (one rounding each), on
    random values over many binades, FP16 subnormals, and exact ties."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100000) * np.exp2(rng.integers(-40, 12, 100000))).astype(np.float32)
    sub = (rng.uniform(-1, 1, 20000) * 2.0 ** -14).astype(np.float32)              # FP16 subnormal range
    for out, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        grid = torch.from_numpy(x).to(tdt).double().numpy()
        step = grid_round(np.abs(grid) * (1 + 2.0 ** -(P[out] + 1)), out, True) - np.abs(grid)
        ties = (np.abs(grid) + step / 2) * np.sign(grid)                            # halfway to the next point
        ties = ties[np.abs(ties) < (6e4 if out == "f16" else 1e30)].astype(np.float32)
        assert np.array_equal(ties.astype(np.float64), ties)                        # exact in FP32
        for vals in (x, sub, ties):
            vals = vals[np.abs(vals) < (6.5e4 if out == "f16" else 3e38)]
            want = torch.from_numpy(vals).to(tdt).double().numpy()
            assert np.array_equal(grid_round_nearest(vals.astype(np.float64), out), want), out
    xd = rng.standard_normal(100000) * np.exp2(rng.integers(-60, 60, 100000))
    assert np.array_equal(grid_round_nearest(xd, "f32"), xd.astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_epilogue_gate_rejects_a_cast_that_rounds_up_or_truncates(out):
    """Values a fraction of one grid step above grid points, with an error
    bound b far below the spacing: the round-to-nearest cast passes, and a
    cast that rounds up or truncates fails wherever it differs from it -- one
    grid step off."""
    ulp = 2.0 ** -(P[out] - 1)                                     # spacing in [1, 2)
    frac = np.array([0.1, 0.3, 0.45, 0.55, 0.7, 0.9])
    y = 1.0 + (np.arange(8)[None, :] + frac[:, None]) * ulp         # 6 x 8 values between grid points
    b = 1e-5                                                       # the error bound before the cast
    D = np.full_like(y, b / (1.13 * TOL["fp32"] + 1e-6))           # makes the gate's b exactly this
    args = ("fp32", out, 1.0, 0.0, None, None, "none")
    rn, up, down = grid_round_nearest(y, out), grid_round(y, out, True), grid_round(y, out, False)
    assert epilogue_check(rn, y, D, *args)[0] <= 1.0
    assert np.any(up != rn) and np.any(down != rn)
    assert epilogue_check(up, y, D, *args)[0] > 1.0
    assert epilogue_check(down, y, D, *args)[0] > 1.0
    # a single element 0.9 grid steps above y (rounded up from 0.1 of a step) fails on its own
    one = rn.copy()
    one[0, 0] = up[0, 0]
    assert one[0, 0] - y[0, 0] > 0.85 * ulp
    assert epilogue_check(one, y, D, *args)[0] > 1.0
    # and a value within b of a midpoint may go either way
    mid = 1.0 + 0.5 * ulp + 0.3 * b
    y2, D2 = np.array([[mid]]), np.array([[D[0, 0]]])
    for c in (1.0, 1.0 + ulp):
        assert epilogue_check(np.array([[c]]), y2, D2, *args)[0] <= 1.0


# ------------------------------------------------------ TF32 input rounding --
# The diagnostic TF32 oracles take their inputs through tf32_round.  Pinned by
# hand-worked ties and by a brute-force nearest-neighbour search in fp64.
from gemm_check import tf32_round


def test_tf32_round_worked_values():
    u = 2.0 ** -10                       # TF32 spacing in [1, 2)
    x = np.array([1.0, 1 + u, 1 + u / 2, 1 + u / 2 + 2 ** -23, 1 + 1.5 * u, 2 - u / 2, -(1 + u / 2 + 2 ** -23)],
                 np.float32)
    rn = [1.0, 1 + u, 1.0, 1 + u, 1 + 2 * u, 2.0, -(1 + u)]       # ties go to the even last bit
    rz = [1.0, 1 + u, 1.0, 1.0, 1 + u, 2 - u, -1.0]
    assert list(tf32_round(x, "rn").astype(np.float64)) == rn
    assert list(tf32_round(x, "rz").astype(np.float64)) == rz


def test_tf32_round_is_nearest_and_toward_zero():
    rng = np.random.default_rng(33)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-60, 60, 200000))).astype(np.float32)
    x[:1000] = rng.integers(-4096, 4096, 1000).astype(np.float32) * np.float32(2.0 ** -11)   # many exact ties
    for mode in ("rn", "rz"):
        r = tf32_round(x, mode)
        assert np.all((r.view(np.uint32) & np.uint32(0x1FFF)) == 0)
    xd = x.astype(np.float64)
    _, e = np.frexp(xd)
    ulp = np.ldexp(1.0, e - 11)                  # TF32 spacing at x (normal inputs)
    lo = np.trunc(xd / ulp) * ulp                # toward zero
    hi = lo + np.sign(xd) * ulp
    assert np.array_equal(tf32_round(x, "rz").astype(np.float64), lo)
    d_lo, d_hi = np.abs(xd - lo), np.abs(hi - xd)
    lo_even = (np.abs(lo / ulp) % 2) == 0
    want = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo_even, lo, hi)))
    assert np.array_equal(tf32_round(x, "rn").astype(np.float64), want)
