"""GPU parity of the fused epilogue (gemm_run_ex) against the fp64 oracle.

C = act(alpha * A.B + beta * C_old + bias) stored as FP32, BF16 or FP16
("Shared memory and tensor cores" section 13.10: bias, activation, residual
add and type cast fused into the GEMM's store).  Every path that writes C is
covered: the SIMT kernel, the tensor-core epilogue warps of every compiled
variant, the split-K reduction and the K = 0 fill; plus the bound check of
gemm_check.epilogue_check, bit-exact small-integer cases, guard bands and
padded leading dimensions, and a full-size BF16 8192^3 case on sampled rows.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300.inputs import C4_BF16_8192, make_epilogue_inputs, make_operands, workload_operands

from gemm_check import (epilogue_check, oracle_c_old, oracle_full, oracle_rows, run_gemm, run_gemm_ex,
                        sample_rows)

pytestmark = pytest.mark.gpu

DTYPES = ("fp32", "tf32", "bf16", "fp16", "e4m3", "e5m2")
OUTS = ("f32", "bf16", "f16")
ACTS = ("none", "relu", "gelu")
OPTION_KEYS = ("tc_bn", "tc_cta_group", "tc_group_m", "tc_max_ctas", "tc_tma_store", "simt_variant", "tc_b_major",
               "debug_stall_mma", "tc_splits", "tc_tail_splits", "tc_tail_halves", "tc_split_reduce", "tc_split_lead")


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


def _check(A, B, dtype, out, alpha, beta, act, seed, with_bias=True, with_old=True, ldc_pad=0):
    M, K = A.shape
    N = B.shape[1]
    c_old, bias = make_epilogue_inputs(M, N, out, seed)
    if not with_old:
        c_old = None
        beta = 0.0
    if not with_bias:
        bias = None
    C = run_gemm_ex(A, B, dtype, out, alpha, beta, c_old, bias, act, ldc_pad=ldc_pad)
    acc, D = oracle_full(A, B, dtype)
    r, _ = epilogue_check(C, acc, D, dtype, out, alpha, beta, c_old, bias, act)
    assert r <= 1.0, f"{dtype}/{out}/{act}: worst error / bound = {r:.3g}"


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("out", OUTS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_epilogue_every_path_output_and_activation(dtype, out, act):
    A, B = make_operands(300, 520, 264, dtype, "normal", seed=31)
    _check(A, B, dtype, out, 0.75, -0.5, act, seed=32)


@pytest.mark.parametrize("dtype", DTYPES)
def test_null_and_identity_epilogue_equal_gemm_run(dtype):
    A, B = make_operands(257, 384, 200, dtype, "uniform", seed=33)
    C0 = run_gemm(A, B, dtype).astype(np.float64)
    assert np.array_equal(run_gemm_ex(A, B, dtype, epilogue=False), C0)
    assert np.array_equal(run_gemm_ex(A, B, dtype, "f32", 1.0, 0.0, None, None, "none"), C0)


@pytest.mark.parametrize("out", ("bf16", "f16"))
@pytest.mark.parametrize("dtype", DTYPES)
def test_small_integers_bit_exact_through_epilogue(dtype, out):
    # |A.B| <= 2*2*32 = 128, |C_old|, |bias| <= 8: every value an integer below
    # 2^8, exact in every output type, so the result is exact.
    M, N, K = 200, 300, 32
    A, B = make_operands(M, N, K, dtype, "ints", seed=34, lo_hi=2)
    gen = torch.Generator().manual_seed(35)
    c_old = torch.randint(-8, 9, (M, N), generator=gen).to(torch.float32)
    bias = torch.randint(-8, 9, (N,), generator=gen).to(torch.float32)
    for act in ("none", "relu"):
        C = run_gemm_ex(A, B, dtype, out, 1.0, -1.0, c_old, bias, act)
        acc, _ = oracle_full(A, B, dtype)
        y = acc - c_old.double().numpy() + bias.double().numpy()[None, :]
        if act == "relu":
            y = np.maximum(y, 0.0)
        assert np.array_equal(C, y)


@pytest.mark.parametrize("store", ("tma", "plain"))
@pytest.mark.parametrize("out", ("f32", "bf16", "f16"))
@pytest.mark.parametrize("cg,bn", [(1, 64), (1, 128), (1, 256), (2, 256)])
@pytest.mark.parametrize("dtype", ("bf16", "tf32", "fp16", "e4m3"))
def test_epilogue_every_tensor_core_variant(dtype, cg, bn, out, store):
    """Every compiled tile with the epilogue in registers ahead of a TMA store
    (old C loaded by TMA) and on the lane = column plain-store path."""
    tg.gemm_set_option("tc_cta_group", cg)
    tg.gemm_set_option("tc_bn", bn)
    tg.gemm_set_option("tc_tma_store", 2 if store == "plain" else 0)
    A, B = make_operands(520, 600, 320, dtype, "normal", seed=36)
    _check(A, B, dtype, out, 1.5, 0.25, "gelu", seed=37)


@pytest.mark.parametrize("splits,tail", [(3, 0), (0, 2)])
@pytest.mark.parametrize("dtype", ("bf16", "tf32", "fp16", "e5m2"))
def test_epilogue_after_split_k_reduction(dtype, splits, tail):
    if splits:
        tg.gemm_set_option("tc_splits", splits)
    else:
        tg.gemm_set_option("tc_tail_splits", tail)
        tg.gemm_set_option("tc_max_ctas", 7)      # 54 tiles on 7 CTAs: a partly idle last round to split
    M, N, K = 700, 520, 2048
    A, B = make_operands(M, N, K, dtype, "normal", seed=38)
    plan = tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N)
    assert plan.tail_tiles > 0 and plan.splits > 1
    _check(A, B, dtype, "f16", -0.5, 1.0, "relu", seed=39)


@pytest.mark.parametrize("splits", (2, 4))
@pytest.mark.parametrize("store", ("tma", "plain"))
@pytest.mark.parametrize("out", ("f32", "bf16"))
@pytest.mark.parametrize("dtype", ("bf16", "tf32", "fp16", "e4m3"))
def test_epilogue_after_split_k_in_cluster_shared_memory(dtype, out, store, splits):
    """The K ranges summed across a cluster, then the whole epilogue (alpha,
    the old C, bias, GELU, the output cast) by the owning CTA's warps, with
    TMA stores and with ordinary stores."""
    for k, v in (("tc_cta_group", 1), ("tc_bn", 128), ("tc_splits", splits), ("tc_split_reduce", 2),
                 ("tc_tma_store", 2 if store == "plain" else 0)):
        tg.gemm_set_option(k, v)
    M, N, K = 300, 520, 2048
    plan = tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N)
    assert plan.cluster_split == splits and plan.splits == splits
    A, B = make_operands(M, N, K, dtype, "normal", seed=40)
    _check(A, B, dtype, out, -0.5, 1.0, "gelu", seed=41)


@pytest.mark.parametrize("splits", (2, 4))
@pytest.mark.parametrize("dtype", ("bf16", "tf32"))
def test_small_integers_bit_exact_through_cluster_split_epilogue(dtype, splits):
    M, N, K = 200, 300, 256
    A, B = make_operands(M, N, K, dtype, "ints", seed=42, lo_hi=1)      # |A.B| <= 256
    gen = torch.Generator().manual_seed(43)
    c_old = torch.randint(-8, 9, (M, N), generator=gen).to(torch.float32)
    bias = torch.randint(-8, 9, (N,), generator=gen).to(torch.float32)
    for k, v in (("tc_cta_group", 1), ("tc_bn", 64), ("tc_splits", splits), ("tc_split_reduce", 2)):
        tg.gemm_set_option(k, v)
    assert tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).cluster_split == splits
    C = run_gemm_ex(A, B, dtype, "f32", 1.0, -1.0, c_old, bias, "relu")
    acc, _ = oracle_full(A, B, dtype)
    assert np.array_equal(C, np.maximum(acc - c_old.double().numpy() + bias.double().numpy()[None, :], 0.0))


@pytest.mark.parametrize("store", ("tma", "plain"))
@pytest.mark.parametrize("out", ("f32", "bf16"))
@pytest.mark.parametrize("dtype", ("bf16", "tf32"))
def test_epilogue_on_column_halves(dtype, out, store):
    """The last round's tiles run as column halves: each half applies bias,
    residual and activation to its own columns (1998 x 1440 on 20 CTA pairs:
    48 tiles, the right-hand column's 8 as halves, one of them part empty)."""
    tg.gemm_set_option("tc_cta_group", 2)
    tg.gemm_set_option("tc_max_ctas", 40)
    tg.gemm_set_option("tc_tail_halves", 2)
    tg.gemm_set_option("tc_tma_store", 2 if store == "plain" else 0)
    M, N, K = 1998, 1440, 512
    A, B = make_operands(M, N, K, dtype, "normal", seed=42)
    assert tg.gemm_plan(M, N, K, tg.DTYPES[dtype], 0, K, 0, N, 0, N).half_tiles == 8
    _check(A, B, dtype, out, 0.75, -0.5, "gelu", seed=43)


@pytest.mark.parametrize("splits", (2, 8))
@pytest.mark.parametrize("out", ("f32", "bf16"))
def test_fp32_epilogue_after_simt_split_k(out, splits):
    """FP32 K cut into ranges: the second kernel applies alpha, the residual,
    the bias and the activation once, to the in-order sum of the ranges."""
    tg.gemm_set_option("simt_splits", splits)
    try:
        A, B = make_operands(333, 257, 515, "fp32", "normal", seed=49)
        _check(A, B, "fp32", out, 0.5, -0.75, "gelu", seed=50, ldc_pad=1)
    finally:
        tg.gemm_set_option("simt_splits", 0)


@pytest.mark.parametrize("out", OUTS)
def test_epilogue_with_k_zero(out):
    M, N = 70, 90
    A, B = make_operands(M, N, 0, "bf16", "normal", seed=40)
    _check(A, B, "bf16", out, 2.0, 0.5, "gelu", seed=41)


@pytest.mark.parametrize("out", OUTS)
@pytest.mark.parametrize("dtype", ("fp32", "bf16"))
def test_epilogue_padded_ldc_and_guards(dtype, out):
    A, B = make_operands(333, 257, 129, dtype, "uniform", seed=42)
    _check(A, B, dtype, out, 1.0, 1.0, "none", seed=43, ldc_pad=3)


@pytest.mark.parametrize("dtype", ("fp32", "bf16"))
def test_epilogue_bias_only_and_residual_only(dtype):
    A, B = make_operands(260, 384, 192, dtype, "normal", seed=44)
    _check(A, B, dtype, "f32", 1.0, 0.0, "relu", seed=45, with_old=False)
    _check(A, B, dtype, "bf16", 1.0, 1.0, "none", seed=46, with_bias=False)


def test_alpha_zero_copies_the_old_c():
    A, B = make_operands(130, 250, 64, "bf16", "normal", seed=47)
    c_old, _ = make_epilogue_inputs(130, 250, "bf16", 48)
    C = run_gemm_ex(A, B, "bf16", "bf16", 0.0, 1.0, c_old, None, "none")
    assert np.array_equal(C, c_old.double().numpy())


def test_rejects_bad_epilogue_arguments():
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    host_bias = torch.zeros(64, dtype=torch.float32)
    ep = tg.make_epilogue(1.0, 0.0, host_bias.data_ptr(), "gelu", "bf16")
    rc = tg.gemm_run_ex(64, 64, 64, tg.GEMM_BF16, A.data_ptr(), 64, A.data_ptr(), 64, C.data_ptr(), 64, ep, s)
    assert rc == tg.GEMM_ERR_INVALID_ARG and "bias" in tg.gemm_last_error()
    ep = tg.make_epilogue(1.0, 0.0, C.data_ptr() + 64, "none", "bf16")
    rc = tg.gemm_run_ex(64, 64, 64, tg.GEMM_BF16, A.data_ptr(), 64, A.data_ptr(), 64, C.data_ptr(), 64, ep, s)
    assert rc == tg.GEMM_ERR_INVALID_ARG and "overlaps" in tg.gemm_last_error()


def test_full_size_bf16_8192_gelu_bias_bf16_out_sampled():
    """The benchmark's fused configuration, automatic plan, checked on sampled rows."""
    w = C4_BF16_8192
    A, B = workload_operands(w)
    c_old, bias = make_epilogue_inputs(w.M, w.N, "bf16", w.seed)
    a, b = A.cuda(), B.cuda()
    C = tg.gemm_ex(a, b, bias=bias.cuda(), act="gelu", out="bf16")
    assert tg.gemm_get_status(torch.cuda.current_stream().cuda_stream) == tg.GEMM_OK
    rows = sample_rows(w.M, tile=256, extra=6, seed=5)
    acc, D = oracle_rows(A, B, "bf16", rows)
    got = C[rows].double().cpu().numpy()
    r, _ = epilogue_check(got, acc, D, "bf16", "bf16", 1.0, 0.0, None, bias, "gelu")
    assert r <= 1.0, f"worst error / bound = {r:.3g}"
    del c_old
