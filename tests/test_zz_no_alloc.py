"""gemm_run_tf32_static, the TF32 GEMM that allocates no device memory,
checked against gemm_run through the C ABI.

The entry point is for callers that cannot allocate device memory while they
run (for example a process whose own allocator already holds all free device
memory): the transposed copy of B that gemm_run puts in a per-call workspace
lives instead in one fixed array the library reserves on each GPU.  Two calls
in a row, with different shapes and inputs, must each agree with gemm_run
within the TF32 tolerance of the other tests; the second call also shows that
the contents the first call left in the shared array do not leak into it.

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


def _both(lib, M, N, K, seed):
    A, B = make_operands(M, N, K, "tf32", "normal", seed)
    a_keep, a_ptr, lda = to_device(A)
    b_keep, b_ptr, ldb = to_device(B)
    c_ref = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    c_new = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gemm_run(M, N, K, tg.GEMM_TF32, a_ptr, lda, b_ptr, ldb, c_ref.data_ptr(), N, stream)
    assert rc == tg.GEMM_OK, tg.gemm_last_error()
    rc = lib.gemm_run_tf32_static(M, N, K, a_ptr, lda, b_ptr, ldb, c_new.data_ptr(), N, stream)
    assert rc == tg.GEMM_OK, tg.gemm_last_error()
    assert lib.gemm_get_status(stream) == tg.GEMM_OK, tg.gemm_last_error()
    _, D = oracle_full(A, B, "tf32")
    del a_keep, b_keep
    return c_new.cpu().numpy(), c_ref.cpu().numpy().astype(np.float64), D


def test_static_scratch_matches_gemm_run_twice(lib):
    for (M, N, K, seed) in ((1000, 1100, 900, 21), (513, 1500, 1028, 22)):
        c_new, c_ref, D = _both(lib, M, N, K, seed)
        assert np.all(np.isfinite(c_new))
        r = error_ratio(c_new, c_ref, D)
        assert r <= TOL["tf32"], (M, N, K, r)


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
