"""Maximum sizes: outputs of more than 2^31 elements, so that every element
offset in the store paths (TMA stores, ordinary stores, the fused epilogue,
the split-K reductions, the SIMT kernel) must be 64-bit.  K is short to keep
the runs quick; rows past the 2^31-element mark are checked against the
oracle one by one."""
import numpy as np
import pytest
import torch

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300.inputs import make_epilogue_inputs, make_operands

from gemm_check import TOL, epilogue_check, error_ratio, oracle_rows

pytestmark = pytest.mark.gpu

OPTION_KEYS = ("tc_bn", "tc_cta_group", "tc_max_ctas", "tc_tma_store", "tc_splits", "tc_tail_splits", "tc_tail_halves",
               "tc_sched", "simt_splits")

M_BIG = (1 << 18) + 7            # 262151 rows
N_BIG = 8200                     # M_BIG * N_BIG = 2.15e9 > 2^31 elements


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
    torch.cuda.empty_cache()


def _rows(M, N):
    """The first row, rows around the 2^31-element mark, the last rows."""
    mark = (1 << 31) // N
    return sorted({0, mark - 1, mark, mark + 1, M - 2, M - 1})


def _check(C, A, B, dtype, rows):
    got = C[rows].double().cpu().numpy()
    ref, D = oracle_rows(A, B, dtype, rows)
    assert error_ratio(got, ref, D) <= TOL[dtype]


@pytest.mark.parametrize("store", ("tma", "plain"))
def test_bf16_output_past_2_31_elements(store):
    assert M_BIG * N_BIG > (1 << 31)
    tg.gemm_set_option("tc_tma_store", 2 if store == "plain" else 0)
    A, B = make_operands(M_BIG, N_BIG, 64, "bf16", "uniform", seed=130)
    C = tg.gemm(A.cuda(), B.cuda())
    assert tg.gemm_get_status(torch.cuda.current_stream().cuda_stream) == tg.GEMM_OK
    _check(C, A, B, "bf16", _rows(M_BIG, N_BIG))
    del C


def test_split_k_reduction_past_2_31_elements():
    tg.gemm_set_option("tc_splits", 2)
    A, B = make_operands(M_BIG, N_BIG, 256, "bf16", "uniform", seed=131)
    C = tg.gemm(A.cuda(), B.cuda())
    assert tg.gemm_get_status(torch.cuda.current_stream().cuda_stream) == tg.GEMM_OK
    _check(C, A, B, "bf16", _rows(M_BIG, N_BIG))
    del C


def test_fused_epilogue_past_2_31_elements():
    A, B = make_operands(M_BIG, N_BIG, 64, "bf16", "uniform", seed=132)
    _, bias = make_epilogue_inputs(1, N_BIG, "bf16", 133)
    C = tg.gemm_ex(A.cuda(), B.cuda(), bias=bias.cuda(), act="relu", out="bf16")
    assert tg.gemm_get_status(torch.cuda.current_stream().cuda_stream) == tg.GEMM_OK
    rows = _rows(M_BIG, N_BIG)
    acc, D = oracle_rows(A, B, "bf16", rows)
    r, _ = epilogue_check(C[rows].double().cpu().numpy(), acc, D, "bf16", "bf16", 1.0, 0.0, None, bias, "relu")
    assert r <= 1.0
    del C


def test_simt_fp32_past_2_31_elements():
    A, B = make_operands(M_BIG, N_BIG, 16, "fp32", "uniform", seed=134)
    C = tg.gemm(A.cuda(), B.cuda(), dtype="fp32")
    assert tg.gemm_get_status(torch.cuda.current_stream().cuda_stream) == tg.GEMM_OK
    _check(C, A, B, "fp32", _rows(M_BIG, N_BIG))
    del C


def test_simt_split_k_past_2_31_elements():
    """Two K ranges forced: each range's partial sums fill an M x N slab of the
    workspace (the second starts past 2^31 elements), and the in-order
    reduction reads both and writes C."""
    tg.gemm_set_option("simt_splits", 2)
    A, B = make_operands(M_BIG, N_BIG, 64, "fp32", "uniform", seed=135)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = torch.empty((M_BIG, N_BIG), dtype=torch.float32, device="cuda")
    plan = tg.gemm_plan(M_BIG, N_BIG, 64, tg.GEMM_FP32, Ad.data_ptr(), 64, Bd.data_ptr(), N_BIG, Cd.data_ptr(),
                        N_BIG)
    assert plan.splits == 2
    C = tg.gemm(Ad, Bd, C=Cd, dtype="fp32")
    assert tg.gemm_get_status(torch.cuda.current_stream().cuda_stream) == tg.GEMM_OK
    _check(C, A, B, "fp32", _rows(M_BIG, N_BIG))
    del C, Cd
