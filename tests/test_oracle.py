"""Pins for the fp64 GEMM oracle, each against something other than itself.

No GPU.  Every check here is fixed by the mathematics of C = A.B ("Shared
memory and tensor cores", ml-compiler-from-scratch ch. 13, section 13.1) or by
an independent library routine: identity and permutation products, all-ones
inputs, exact integer arithmetic, a second loop order, float64 matmul, and the
libraries' own BF16 and FP16 conversions.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array, make_operands


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def _bf16_bits(x_float):
    t = torch.as_tensor(np.asarray(x_float, dtype=np.float32)).to(torch.bfloat16)
    return as_oracle_array(t).copy()


def _f16_bits(x_float):
    return np.asarray(x_float, dtype=np.float32).astype(np.float16).view(np.uint16).copy()


@pytest.mark.parametrize("M,N", [(1, 1), (7, 13), (64, 33)])
def test_identity_left(M, N):
    rng = np.random.default_rng(1)
    B = _f32(rng.standard_normal((M, N)))
    C = oracle.gemm(np.eye(M, dtype=np.float32), B)
    assert np.array_equal(C, B.astype(np.float64))


def test_identity_right():
    rng = np.random.default_rng(2)
    A = _f32(rng.standard_normal((19, 23)))
    C = oracle.gemm(A, np.eye(23, dtype=np.float32))
    assert np.array_equal(C, A.astype(np.float64))


def test_permutation():
    rng = np.random.default_rng(3)
    M, N = 37, 29
    perm = rng.permutation(M)
    P = np.zeros((M, M), np.float32)
    P[np.arange(M), perm] = 1.0          # row i of P selects row perm[i] of B
    B = _f32(rng.uniform(-1, 1, (M, N)))
    C = oracle.gemm(P, B)
    assert np.array_equal(C, B[perm].astype(np.float64))
    # and the transposed permutation undoes it: a transposed-operand bug fails here
    C2 = oracle.gemm(_f32(P.T), _f32(C))
    assert np.array_equal(C2, B.astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (5, 9, 17), (33, 65, 129), (16, 16, 4096)])
def test_all_ones_gives_K(M, N, K):
    C, D = oracle.gemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32), with_scale=True)
    assert np.all(C == K) and np.all(D == K)


def test_small_integers_exact_vs_integer_matmul():
    rng = np.random.default_rng(4)
    M, N, K = 45, 38, 300
    Ai = rng.integers(-8, 9, (M, K))
    Bi = rng.integers(-8, 9, (K, N))
    C, D = oracle.gemm(_f32(Ai), _f32(Bi), with_scale=True)
    assert np.array_equal(C, (Ai @ Bi).astype(np.float64))
    assert np.array_equal(D, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


def test_small_integers_exact_bf16():
    rng = np.random.default_rng(5)
    M, N, K = 31, 40, 257
    Ai = rng.integers(-8, 9, (M, K))
    Bi = rng.integers(-8, 9, (K, N))
    C = oracle.gemm(_bf16_bits(Ai), _bf16_bits(Bi), bf16=True)
    assert np.array_equal(C, (Ai @ Bi).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 16, 15), (16, 17, 17)])
def test_second_loop_order_bit_equal(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = _f32(rng.standard_normal((M, K)))
    B = _f32(rng.standard_normal((K, N)))
    assert np.array_equal(oracle.gemm(A, B), oracle.gemm_jik(A, B))
    Ab, Bb = _bf16_bits(A), _bf16_bits(B)
    assert np.array_equal(oracle.gemm(Ab, Bb, bf16=True), oracle.gemm_jik(Ab, Bb, bf16=True))


def test_against_float64_library_matmul():
    rng = np.random.default_rng(6)
    A = _f32(rng.standard_normal((64, 80)))
    B = _f32(rng.standard_normal((80, 48)))
    C, D = oracle.gemm(A, B, with_scale=True)
    ref = (torch.from_numpy(A).double() @ torch.from_numpy(B).double()).numpy()
    assert np.max(np.abs(C - ref) / D) < 1e-14


def test_bf16_widening_matches_library_conversion():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen_bf16(bits)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    # a few fixed patterns: 1.0, -2.0, the largest finite value, +inf
    assert list(oracle.widen_bf16(np.array([0x3F80, 0xC000, 0x7F7F, 0x7F80], np.uint16))) == [
        1.0, -2.0, float(np.float32(3.3895313892515355e38)), float("inf")]


def test_leading_dimensions_honoured():
    A, B = make_operands(21, 18, 27, "fp32", "ints", 7, lda_pad=5, ldb_pad=3)
    a, b = as_oracle_array(A), as_oracle_array(B)
    assert a.strides[0] == (27 + 5) * 4 and b.strides[0] == (18 + 3) * 4
    C = oracle.gemm(a, b)                 # the NaN padding must never be read
    assert np.all(np.isfinite(C))
    assert np.array_equal(C, np.ascontiguousarray(a).astype(np.int64) @ np.ascontiguousarray(b).astype(np.int64))


def test_rows_variant_matches_full():
    A, B = make_operands(50, 40, 60, "bf16", "normal", 8)
    a, b = as_oracle_array(A), as_oracle_array(B)
    C, D = oracle.gemm(a, b, bf16=True, with_scale=True)
    rows = [0, 7, 49, 23]
    Cr, Dr = oracle.gemm_rows(a, b, rows, bf16=True)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Dr, D[rows])


def test_rows_variant_f32_matches_full():
    # rows in any order, repeated, first and last; padded leading dimensions
    A, B = make_operands(41, 30, 52, "fp32", "normal", 12, lda_pad=3, ldb_pad=2)
    a, b = as_oracle_array(A), as_oracle_array(B)
    C, D = oracle.gemm(a, b, with_scale=True)
    rows = [40, 3, 3, 0, 17]
    Cr, Dr = oracle.gemm_rows(a, b, rows)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(Dr, D[rows])


def test_empty_sum_and_empty_shapes():
    C = oracle.gemm(np.zeros((4, 0), np.float32), np.zeros((0, 6), np.float32))
    assert C.shape == (4, 6) and np.all(C == 0)
    assert oracle.gemm(np.zeros((0, 3), np.float32), np.zeros((3, 5), np.float32)).shape == (0, 5)


def test_threads_reported():
    assert oracle.num_threads() >= 1


def test_f16_widening_matches_library_conversion():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen_f16(bits)
    lib = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    # 1.0, -2.0, the largest finite value, the smallest subnormal, +inf
    assert list(oracle.widen_f16(np.array([0x3C00, 0xC000, 0x7BFF, 0x0001, 0x7C00], np.uint16))) == [
        1.0, -2.0, 65504.0, 2.0 ** -24, float("inf")]


def test_small_integers_exact_f16():
    rng = np.random.default_rng(9)
    M, N, K = 29, 43, 300
    Ai = rng.integers(-8, 9, (M, K))
    Bi = rng.integers(-8, 9, (K, N))
    C, D = oracle.gemm(_f16_bits(Ai), _f16_bits(Bi), fp16=True, with_scale=True)
    assert np.array_equal(C, (Ai @ Bi).astype(np.float64))
    assert np.array_equal(D, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 16, 15)])
def test_f16_second_loop_order_and_library(M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = _f16_bits(rng.standard_normal((M, K)))
    B = _f16_bits(rng.standard_normal((K, N)))
    C = oracle.gemm(A, B, fp16=True)
    assert np.array_equal(C, oracle.gemm_jik(A, B, fp16=True))
    ref = A.view(np.float16).astype(np.float64) @ B.view(np.float16).astype(np.float64)
    assert np.allclose(C, ref, rtol=1e-13, atol=1e-13)
    r, _ = oracle.gemm_rows(A, B, [M - 1], fp16=True)
    assert np.array_equal(r[0], C[M - 1])


# ---------------------------------------------------------------- epilogue --
# Pins for the fused epilogue ("Shared memory and tensor cores" section 13.10:
# bias, activation, residual add, type cast on the accumulator), each against
# a library routine, printed values of the normal CDF, or an identity.

def test_epilogue_default_is_the_product():
    acc = np.random.default_rng(20).standard_normal((9, 14))
    assert np.array_equal(oracle.epilogue(acc), acc)


@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_epilogue_against_library_addmm_and_activation(act):
    rng = np.random.default_rng(21)
    M, N, K = 23, 17, 40
    Ai = rng.integers(-6, 7, (M, K))
    Bi = rng.integers(-6, 7, (K, N))
    c_old = _f32(rng.standard_normal((M, N)))
    bias = _f32(rng.standard_normal(N))
    alpha, beta = 0.37, -1.25
    acc = oracle.gemm(_f32(Ai), _f32(Bi))
    y = oracle.epilogue(acc, alpha, beta, c_old, "f32", bias, act)
    t = torch.addmm(torch.from_numpy(c_old).double(), torch.from_numpy(Ai).double(), torch.from_numpy(Bi).double(),
                    beta=beta, alpha=alpha) + torch.from_numpy(bias).double()
    if act == "relu":
        t = torch.relu(t)
    elif act == "gelu":
        t = torch.nn.functional.gelu(t)            # the erf form
    assert np.allclose(y, t.numpy(), rtol=1e-13, atol=1e-13)


def test_epilogue_gelu_printed_normal_cdf_values():
    # Phi(1), Phi(-1), Phi(2), Phi(3) as printed in standard normal tables.
    x = np.array([[0.0, 1.0, -1.0, 2.0, 3.0]])
    y = oracle.epilogue(x, act="gelu")
    ref = [0.0, 0.8413447460685429, -0.15865525393145707, 2 * 0.9772498680518208, 3 * 0.9986501019683699]
    assert np.allclose(y[0], ref, rtol=1e-14, atol=0)


def test_epilogue_gelu_odd_part_is_half_identity():
    # Phi(-x) = 1 - Phi(x), so GELU(x) - GELU(-x) = x for every x.
    x = np.random.default_rng(22).uniform(-6, 6, (4, 50))
    d = oracle.epilogue(x, act="gelu") - oracle.epilogue(-x, act="gelu")
    assert np.allclose(d, x, rtol=1e-14, atol=1e-14)


def test_epilogue_relu_signs():
    pos = np.abs(np.random.default_rng(23).standard_normal((6, 7))) + 0.1
    assert np.array_equal(oracle.epilogue(pos, act="relu"), pos)
    assert np.array_equal(oracle.epilogue(-pos, act="relu"), np.zeros_like(pos))


def test_epilogue_bias_is_per_column():
    M, N = 5, 11                          # M != N: a row-indexed bias would differ
    bias = np.arange(N, dtype=np.float32) - 3.5
    y = oracle.epilogue(np.zeros((M, N)), bias=bias)
    assert np.array_equal(y, np.broadcast_to(bias.astype(np.float64), (M, N)))


@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_epilogue_reads_old_c_in_the_output_type(out):
    vals = np.random.default_rng(24).standard_normal((7, 9)).astype(np.float32)
    if out == "bf16":
        t = torch.from_numpy(vals).to(torch.bfloat16)
        bits = as_oracle_array(t).copy()
        lib = t.double().numpy()
    else:
        bits = _f16_bits(vals)
        lib = bits.view(np.float16).astype(np.float64)
    y = oracle.epilogue(np.zeros((7, 9)), alpha=1.0, beta=-2.0, c_old=bits, out=out)
    assert np.array_equal(y, -2.0 * lib)


def test_epilogue_beta_zero_never_reads_old_c():
    acc = np.ones((3, 4))
    assert np.array_equal(oracle.epilogue(acc, alpha=3.0, beta=0.0, c_old=None), 3.0 * acc)


# -------------------------------------------------------------------- FP8 --
# Pins for the FP8 (OCP E4M3 and E5M2) widening and products: every byte
# against the library's own FP8 types, printed format constants, exact
# integer products, and the second loop order.
FP8_LIB = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _fp8_bytes(x_float, fmt):
    t = torch.as_tensor(np.asarray(x_float, dtype=np.float32)).to(FP8_LIB[fmt])
    return as_oracle_array(t).copy()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_widening_matches_library_conversion(fmt):
    bits = np.arange(256, dtype=np.uint8)
    ours = oracle.widen_fp8(bits, fmt)
    lib = torch.from_numpy(bits).view(FP8_LIB[fmt]).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])


def test_fp8_format_constants():
    # E4M3: 1.0, the largest finite value 448, the smallest subnormal 2^-9, the only NaN pattern
    e4 = oracle.widen_fp8(np.array([0x38, 0x7E, 0x01, 0xB8, 0x7F], np.uint8), "e4m3")
    assert list(e4[:4]) == [1.0, 448.0, 2.0 ** -9, -1.0] and np.isnan(e4[4])
    # E5M2: 1.0, the largest finite value 57344, the smallest subnormal 2^-16, +inf
    e5 = oracle.widen_fp8(np.array([0x3C, 0x7B, 0x01, 0x7C], np.uint8), "e5m2")
    assert list(e5) == [1.0, 57344.0, 2.0 ** -16, float("inf")]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_small_integers_exact_fp8(fmt):
    # integers up to 8 are exact in both formats
    rng = np.random.default_rng(10)
    M, N, K = 27, 41, 333
    Ai = rng.integers(-8, 9, (M, K))
    Bi = rng.integers(-8, 9, (K, N))
    C, D = oracle.gemm(_fp8_bytes(Ai, fmt), _fp8_bytes(Bi, fmt), fp8=fmt, with_scale=True)
    assert np.array_equal(C, (Ai @ Bi).astype(np.float64))
    assert np.array_equal(D, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 16, 15)])
def test_fp8_second_loop_order_library_and_rows(fmt, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    A = _fp8_bytes(rng.standard_normal((M, K)), fmt)
    B = _fp8_bytes(rng.standard_normal((K, N)), fmt)
    C = oracle.gemm(A, B, fp8=fmt)
    assert np.array_equal(C, oracle.gemm_jik(A, B, fp8=fmt))
    lib = (torch.from_numpy(A).view(FP8_LIB[fmt]).double() @ torch.from_numpy(B).view(FP8_LIB[fmt]).double()).numpy()
    assert np.allclose(C, lib, rtol=1e-13, atol=1e-13)
    r, _ = oracle.gemm_rows(A, B, [M - 1, 0], fp8=fmt)
    assert np.array_equal(r, C[[M - 1, 0]])
