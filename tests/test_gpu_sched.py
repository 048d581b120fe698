"""GPU parity under the dynamic schedule (Cluster Launch Control, "Learn
CuTeDSL" section 8.2): one cluster per work unit is launched and the running
clusters steal the units of the ones that have not started.  Every unit must
still be computed exactly once, so the results are bit-identical to the static
schedule's, on every tile, input type, split-K layout, fused epilogue and
grouped launch; small-integer inputs must be exact.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300.inputs import (C4_BF16_8192, GROUPED_BF16, grouped_operands, make_epilogue_inputs,
                                                 make_operands, workload_operands)

from gemm_check import oracle_full, run_gemm, run_gemm_ex

pytestmark = pytest.mark.gpu

OPTION_KEYS = ("tc_bn", "tc_cta_group", "tc_group_m", "tc_max_ctas", "tc_tma_store", "simt_variant", "tc_b_major",
               "debug_stall_mma", "tc_splits", "tc_tail_splits", "tc_tail_halves", "tc_sched")


@pytest.fixture(scope="module", autouse=True)
def lib():
    tgbuild.build()
    tg.load_library()
    yield


@pytest.fixture(autouse=True)
def default_options():
    for k in OPTION_KEYS:
        tg.gemm_set_option(k, 0)
    yield
    for k in OPTION_KEYS:
        tg.gemm_set_option(k, 0)


def _both(fn):
    """fn() under the static, then the dynamic schedule."""
    tg.gemm_set_option("tc_sched", 1)
    a = fn()
    tg.gemm_set_option("tc_sched", 2)
    b = fn()
    tg.gemm_set_option("tc_sched", 0)
    return a, b


def test_dynamic_schedule_smallest_case_first():
    """One small pair-tile GEMM, with a short wait bound, before anything larger."""
    tg.gemm_set_option("wait_timeout_ms", 500)
    try:
        tg.gemm_set_option("tc_sched", 2)
        A, B = make_operands(512, 768, 320, "bf16", "ints", seed=120)
        C = run_gemm(A, B, "bf16")
        ref, _ = oracle_full(A, B, "bf16")
        assert np.array_equal(C, ref)
    finally:
        tg.gemm_set_option("wait_timeout_ms", 2000)


@pytest.mark.parametrize("cg,bn", [(1, 64), (1, 128), (1, 256), (2, 256)])
@pytest.mark.parametrize("dtype", ("bf16", "tf32", "fp16", "e4m3"))
def test_dynamic_equals_static_and_exact(dtype, cg, bn):
    tg.gemm_set_option("tc_cta_group", cg)
    tg.gemm_set_option("tc_bn", bn)
    A, B = make_operands(1300, 1100, 700, dtype, "ints", seed=121)
    s, d = _both(lambda: run_gemm(A, B, dtype))
    ref, _ = oracle_full(A, B, dtype)
    assert np.array_equal(d, ref) and np.array_equal(s, d)


@pytest.mark.parametrize("splits,tail", [(3, 0), (0, 2)])
def test_dynamic_with_split_k(splits, tail):
    A, B = make_operands(700, 520, 2048, "bf16", "normal", seed=122)
    if splits:
        tg.gemm_set_option("tc_splits", splits)
    else:
        tg.gemm_set_option("tc_tail_splits", tail)
        tg.gemm_set_option("tc_max_ctas", 7)
    s, d = _both(lambda: run_gemm(A, B, "bf16"))
    assert np.array_equal(s, d)


def test_dynamic_with_column_halves():
    """The last tiles' column halves are units like any other for the stealer."""
    A, B = make_operands(1998, 1440, 1024, "bf16", "ints", seed=125)
    tg.gemm_set_option("tc_cta_group", 2)
    tg.gemm_set_option("tc_max_ctas", 40)
    assert tg.gemm_plan(1998, 1440, 1024, tg.GEMM_BF16, 0, 1024, 0, 1440, 0, 1440).half_tiles == 8
    s, d = _both(lambda: run_gemm(A, B, "bf16"))
    ref, _ = oracle_full(A, B, "bf16")
    assert np.array_equal(d, ref) and np.array_equal(s, d)


def test_dynamic_with_fused_residual_epilogue():
    A, B = make_operands(1000, 1536, 512, "bf16", "normal", seed=123)
    c_old, bias = make_epilogue_inputs(1000, 1536, "bf16", 124)
    s, d = _both(lambda: run_gemm_ex(A, B, "bf16", "bf16", 0.5, 1.0, c_old, bias, "gelu"))
    assert np.array_equal(s, d)


def test_dynamic_grouped_equals_static():
    w = GROUPED_BF16
    pairs = grouped_operands(w)[:6]
    dev = [(A.cuda(), B.cuda()) for A, B in pairs]
    s, d = _both(lambda: [c.cpu() for c in tg.gemm_grouped([a for a, _ in dev], [b for _, b in dev])])
    for x, y in zip(s, d):
        assert torch.equal(x, y)


def test_dynamic_full_size_bf16_8192_equals_static():
    A, B = workload_operands(C4_BF16_8192)
    a, b = A.cuda(), B.cuda()
    s, d = _both(lambda: tg.gemm(a, b).cpu())
    assert torch.equal(s, d)
