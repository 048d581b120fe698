"""GPU parity of the grouped GEMM (gemm_run_grouped) against the fp64 oracle.

A grouped launch computes a batch of independent GEMMs ("Learn CuTeDSL"
section 8.4); by definition each group's C is that group's own A_g . B_g (with
the shared epilogue and the group's bias), so every group is checked against
the oracle on its own.  Covered: every input type, ragged and degenerate
groups (M = 0, K = 0, 1 x 1 x 1), every compiled tile, packed and plain-store
groups mixed with TMA-addressable ones, the fused epilogue with per-group
bias, bit-equality with the same GEMMs run one by one, and the skewed
16-group workload the benchmark times, on sampled rows.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300.inputs import (GROUPED_BF16, grouped_operands, make_epilogue_inputs,
                                                 make_operands)

from gemm_check import (TOL, epilogue_check, error_ratio, oracle_full, oracle_rows, run_gemm, sample_rows,
                        to_device)

pytestmark = pytest.mark.gpu

OPTION_KEYS = ("tc_bn", "tc_cta_group", "tc_group_m", "tc_max_ctas", "tc_tma_store", "simt_variant", "tc_b_major",
               "debug_stall_mma", "tc_splits", "tc_tail_splits", "tc_tail_halves")
GUARD = 64


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


OUT_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}

# ragged, tiny, empty and long-K groups side by side
SHAPES = [(300, 520, 264), (128, 256, 64), (1000, 64, 999), (1, 1, 1), (0, 77, 50), (257, 129, 130),
          (64, 300, 0), (513, 700, 320)]


def run_grouped(pairs, dtype, out="f32", alpha=1.0, beta=0.0, act="none", c_olds=None, biases=None, ldc_pads=None,
                offsets=None):
    """Runs every (A, B) pair as one grouped launch; each C sits in its own
    NaN-guarded buffer.  Returns the Cs as float64 arrays after checking the
    status word, the guards and the ldc padding."""
    keep, groups, cbufs = [], [], []
    for g, (A, B) in enumerate(pairs):
        M, K = A.shape
        N = B.shape[1]
        off = offsets[g] if offsets else 0
        ka, pa, lda = to_device(A, off)
        kb, pb, ldb = to_device(B)
        ldc = max(N, 1) + (ldc_pads[g] if ldc_pads else 0)
        cbuf = torch.full((2 * GUARD + M * ldc,), float("nan"), dtype=OUT_TORCH[out], device="cuda")
        if c_olds is not None and M and N:
            cbuf[GUARD:GUARD + M * ldc].view(M, ldc)[:, :N].copy_(c_olds[g].to(OUT_TORCH[out]))
        bias = biases[g].cuda() if biases is not None and biases[g] is not None else None
        keep += [ka, kb, bias]
        cbufs.append((cbuf, M, N, ldc))
        groups.append(tg.GemmGroup(M, N, K, pa, lda, pb, ldb, cbuf.data_ptr() + GUARD * cbuf.element_size(), ldc,
                                   bias.data_ptr() if bias is not None else None))
    s = torch.cuda.current_stream().cuda_stream
    ep = tg.make_epilogue(alpha, beta, 0, act, out)
    rc = tg.gemm_run_grouped(tg.DTYPES[dtype], groups, ep, s)
    assert rc == tg.GEMM_OK, tg.gemm_last_error()
    assert tg.gemm_get_status(s) == tg.GEMM_OK, tg.gemm_last_error()
    outs = []
    for cbuf, M, N, ldc in cbufs:
        h = cbuf.cpu().double().numpy()
        assert np.all(np.isnan(h[:GUARD])) and np.all(np.isnan(h[GUARD + M * ldc:])), "write outside C"
        C = h[GUARD:GUARD + M * ldc].reshape(M, ldc)
        assert np.all(np.isnan(C[:, N:])), "write into the ldc padding"
        outs.append(C[:, :N].copy())
    del keep
    return outs


@pytest.mark.parametrize("dtype", ("bf16", "fp16", "tf32", "e4m3", "e5m2", "fp32"))
def test_grouped_small_integers_bit_exact(dtype):
    pairs = [make_operands(M, N, K, dtype, "ints", seed=50 + g) for g, (M, N, K) in enumerate(SHAPES)]
    Cs = run_grouped(pairs, dtype)
    for (A, B), C in zip(pairs, Cs):
        ref, _ = oracle_full(A, B, dtype)
        assert np.array_equal(C, ref)


@pytest.mark.parametrize("cg,bn", [(1, 64), (1, 128), (1, 256), (2, 256)])
@pytest.mark.parametrize("dtype", ("bf16", "tf32", "e4m3"))
def test_grouped_every_tile_and_few_ctas(dtype, cg, bn):
    pairs = [make_operands(M, N, K, dtype, "ints", seed=60 + g) for g, (M, N, K) in enumerate(SHAPES)]
    tg.gemm_set_option("tc_cta_group", cg)
    tg.gemm_set_option("tc_bn", bn)
    for max_ctas in (0, 2 * cg):           # the whole machine, then several units per CTA
        tg.gemm_set_option("tc_max_ctas", max_ctas)
        Cs = run_grouped(pairs, dtype)
        for (A, B), C in zip(pairs, Cs):
            ref, _ = oracle_full(A, B, dtype)
            assert np.array_equal(C, ref)


@pytest.mark.parametrize("dtype", ("bf16", "e4m3"))
def test_grouped_packed_and_plain_store_groups(dtype):
    """Misaligned A (packed), ragged pitches and C not addressable by TMA in some
    groups, next to groups that need none of that."""
    shapes = [(200, 256, 128), (199, 301, 129), (256, 257, 64), (130, 512, 96)]
    pairs = [make_operands(M, N, K, dtype, "ints", seed=70 + g, lda_pad=p, ldb_pad=p)
             for g, ((M, N, K), p) in enumerate(zip(shapes, (0, 3, 0, 5)))]
    Cs = run_grouped(pairs, dtype, ldc_pads=[0, 1, 3, 0], offsets=[0, 1, 0, 2])
    for (A, B), C in zip(pairs, Cs):
        ref, _ = oracle_full(A, B, dtype)
        assert np.array_equal(C, ref)


@pytest.mark.parametrize("out,act", [("bf16", "gelu"), ("f32", "relu"), ("f16", "none")])
@pytest.mark.parametrize("dtype", ("bf16", "fp16", "fp32"))
def test_grouped_fused_epilogue_with_per_group_bias(dtype, out, act):
    shapes = [(300, 520, 264), (129, 256, 200), (64, 128, 0), (513, 320, 96)]
    pairs = [make_operands(M, N, K, dtype, "normal", seed=80 + g) for g, (M, N, K) in enumerate(shapes)]
    olds, biases = [], []
    for g, (M, N, K) in enumerate(shapes):
        c_old, bias = make_epilogue_inputs(M, N, out, 90 + g)
        olds.append(c_old)
        biases.append(bias if g != 1 else None)           # one group without a bias
    Cs = run_grouped(pairs, dtype, out, 0.75, -0.5, act, olds, biases)
    for (A, B), C, c_old, bias in zip(pairs, Cs, olds, biases):
        acc, D = oracle_full(A, B, dtype)
        r, _ = epilogue_check(C, acc, D, dtype, out, 0.75, -0.5, c_old, bias, act)
        assert r <= 1.0, r


@pytest.mark.parametrize("dtype", ("bf16", "tf32"))
def test_grouped_equals_the_same_gemms_one_by_one(dtype):
    """With the tile forced to match, a group's C is bit-identical to gemm_run's:
    same tiles, same K order, no split."""
    shapes = [(1000, 1000, 1000), (257, 513, 777), (2048, 256, 1500)]
    pairs = [make_operands(M, N, K, dtype, "normal", seed=100 + g) for g, (M, N, K) in enumerate(shapes)]
    tg.gemm_set_option("tc_cta_group", 1)
    tg.gemm_set_option("tc_bn", 128)
    tg.gemm_set_option("tc_splits", 1)
    Cs = run_grouped(pairs, dtype)
    for (A, B), C in zip(pairs, Cs):
        assert np.array_equal(C, run_gemm(A, B, dtype).astype(np.float64))


def test_grouped_workload_sampled_rows():
    """The benchmark's skewed 16-group BF16 workload, automatic plan."""
    w = GROUPED_BF16
    pairs = grouped_operands(w)
    dev = [(A.cuda(), B.cuda()) for A, B in pairs]
    Cs = tg.gemm_grouped([a for a, _ in dev], [b for _, b in dev])
    assert tg.gemm_get_status(torch.cuda.current_stream().cuda_stream) == tg.GEMM_OK
    for g in (0, 6, 7, 15):                       # the smallest, the two largest, the last
        A, B = pairs[g]
        rows = sample_rows(A.shape[0], extra=4, seed=g)
        ref, D = oracle_rows(A, B, "bf16", rows)
        got = Cs[g][rows].cpu().numpy()
        assert error_ratio(got, ref, D) <= TOL["bf16"]
