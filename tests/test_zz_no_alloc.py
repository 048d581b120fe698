"""gemm_run_tf32_static, the TF32 GEMM that allocates no device memory,
checked against the fp64 oracle through the C ABI.

The entry point is for callers that cannot allocate device memory while they
run (for example a process whose own allocator already holds all free device
memory): the transposed copy of B that gemm_run puts in a per-call workspace
lives instead in one fixed array the library reserves on each GPU.  Every call
shares that array and it keeps the previous call's contents, so these tests
check what that sharing could break:

* two calls in a row with different shapes and random inputs, each within the
  TF32 bound of the oracle, and a small-integer case that must be bit-exact;
* a chain of eight calls on one stream with no host synchronisation between
  them, each with its own B: call i + 1 rewrites the array while call i's GEMM
  may still be reading it unless the launch order holds, so every result must
  be exact;
* a call whose K is not a multiple of 4 after a call that filled the whole
  array with NaN: the padding columns of the transposed copy then hold the
  earlier NaN and must never be read.

This file is collected last, so a run that stops at the first failure has
already run every other test.  It also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300.inputs import make_operands

from gemm_check import TOL, error_ratio, oracle_full, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    tgbuild.build()
    lib = tg.load_library()
    for k in ("tc_bn", "tc_cta_group", "tc_group_m", "tc_max_ctas", "tc_tma_store", "simt_variant", "tc_b_major",
              "tc_splits"):
        tg.gemm_set_option(k, 0)
    return lib


def _static(lib, A, B, stream=None, sync=True):
    """C = A.B through gemm_run_tf32_static; returns (C on the device, keepalives)."""
    M, K = A.shape
    N = B.shape[1]
    a_keep, a_ptr, lda = to_device(A)
    b_keep, b_ptr, ldb = to_device(B)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = lib.gemm_run_tf32_static(M, N, K, a_ptr, lda, b_ptr, ldb, C.data_ptr(), N, s)
    assert rc == tg.GEMM_OK, tg.gemm_last_error()
    if sync:
        assert lib.gemm_get_status(s) == tg.GEMM_OK, tg.gemm_last_error()
    return C, (a_keep, b_keep)


def test_static_scratch_matches_the_oracle_twice(lib):
    for (M, N, K, seed) in ((1000, 1100, 900, 21), (513, 1500, 1028, 22)):
        A, B = make_operands(M, N, K, "tf32", "normal", seed)
        C, keep = _static(lib, A, B)
        c = C.cpu().numpy()
        assert np.all(np.isfinite(c))
        Cref, D = oracle_full(A, B, "tf32")
        r = error_ratio(c, Cref, D)
        assert r <= TOL["tf32"], (M, N, K, r)


def test_static_scratch_small_integers_bit_exact(lib):
    # integers in [-8, 8]: TF32 holds them exactly and every sum is an exact FP32 integer
    A, B = make_operands(300, 700, 1000, "tf32", "ints", 24)
    C, keep = _static(lib, A, B)
    Cref, _ = oracle_full(A, B, "tf32")
    assert np.array_equal(C.cpu().numpy().astype(np.float64), Cref)


def test_static_scratch_chain_without_host_sync(lib):
    """Eight calls back to back on one stream, each with its own B: each call's
    transpose rewrites the shared array that the previous call's GEMM reads,
    so only the launch order keeps them apart."""
    M, N, K = 384, 1536, 640
    A, _ = make_operands(M, N, K, "tf32", "ints", 25)
    Bs = [make_operands(M, N, K, "tf32", "ints", 100 + i)[1] for i in range(8)]
    stream = torch.cuda.current_stream().cuda_stream
    outs = [_static(lib, A, B, stream, sync=False) for B in Bs]
    assert lib.gemm_get_status(stream) == tg.GEMM_OK, tg.gemm_last_error()
    for i, ((C, _), B) in enumerate(zip(outs, Bs)):
        Cref, _ = oracle_full(A, B, "tf32")
        assert np.array_equal(C.cpu().numpy().astype(np.float64), Cref), f"call {i} of the chain"


def test_static_scratch_padding_left_over_from_an_earlier_call_is_not_read(lib):
    # First call: N x K = 2048 x 2048 fills the whole array (4 Mi floats) with the
    # transpose of a NaN B (its C is NaN and not checked).
    A0 = torch.ones((64, 2048), dtype=torch.float32)
    B0 = torch.full((2048, 2048), float("nan"), dtype=torch.float32)
    C0, keep0 = _static(lib, A0, B0)
    # Second call: K = 1027, so the transposed rows have a padding column (pitch
    # 1028) that still holds NaN; A has its leading dimension padded to 1028
    # (the entry point cannot copy A to make its pitch a multiple of 4).
    A, B = make_operands(300, 1500, 1027, "tf32", "normal", 26, lda_pad=1)
    assert A.stride(0) == 1028
    C, keep = _static(lib, A, B)
    c = C.cpu().numpy()
    assert np.all(np.isfinite(c))
    Cref, D = oracle_full(A, B, "tf32")
    r = error_ratio(c, Cref, D)
    assert r <= TOL["tf32"], r


def test_static_scratch_rejects_what_it_cannot_serve(lib):
    n = 4096   # N * roundup(K, 4) = 16 Mi floats > 4 Mi floats of scratch
    rc = lib.gemm_run_tf32_static(n, n, n, 1 << 30, n, 1 << 31, n, 1 << 32, n, 0)
    assert rc == tg.GEMM_ERR_INVALID_ARG
    assert "static scratch" in tg.gemm_last_error()
    assert tg.TF32_STATIC_SCRATCH_BYTES == 16 * 1024 * 1024
    # an A row pitch of 4108 bytes would need a copy of A, for which there is no scratch
    A, B = make_operands(64, 96, 1027, "tf32", "normal", 23)
    a_keep, a_ptr, lda = to_device(A)
    b_keep, b_ptr, ldb = to_device(B)
    c = torch.empty((64, 96), dtype=torch.float32, device="cuda")
    rc = lib.gemm_run_tf32_static(64, 96, 1027, a_ptr, lda, b_ptr, ldb, c.data_ptr(), 96,
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == tg.GEMM_ERR_UNSUPPORTED and "copy of A" in tg.gemm_last_error()
