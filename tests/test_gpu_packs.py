"""Operands whose pitch or base TMA cannot address are first packed into a
stream-ordered workspace with a 16-byte pitch.  Checked here: exact on small
integers against the oracle with A only, B only or both packed, padded
pitches and odd base addresses, for 16-bit, TF32 and FP8 inputs; and
back-to-back calls with no host synchronisation, each with its own
workspace from the stream-ordered pool."""
import numpy as np
import pytest
import torch

import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300.inputs import make_operands

from gemm_check import oracle_full, run_gemm

pytestmark = pytest.mark.gpu

ELEM = {"bf16": 2, "fp16": 2, "tf32": 4, "e4m3": 1}


@pytest.fixture(scope="module", autouse=True)
def lib():
    tgbuild.build()
    tg.load_library()
    for k in ("tc_sched", "tc_b_major", "tc_bn", "tc_cta_group"):
        tg.gemm_set_option(k, 0)
    yield


def _padded(x, pad):
    """The same values in a buffer whose rows are `pad` elements longer."""
    rows, cols = x.shape
    buf = torch.zeros((rows, cols + pad), dtype=x.dtype)
    buf[:, :cols] = x
    return buf[:, :cols]


CASES = [  # M, N, K, A pitch pad, B pitch pad, A base offset, B base offset (elements)
    (300, 700, 1100, 0, 0, 0, 0),
    (129, 257, 65, 0, 0, 0, 0),
    (256, 512, 1001, 0, 0, 0, 0),
    (1000, 1001, 512, 0, 0, 0, 0),
    (40, 1000, 777, 0, 0, 1, 3),
    (2049, 3071, 2051, 0, 0, 0, 0),
    (512, 640, 384, 3, 5, 0, 0),
    (1, 17, 9, 0, 0, 0, 0),
]


@pytest.mark.parametrize("dtype", ("bf16", "fp16", "tf32", "e4m3"))
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:3])) + ("_pad" if c[3] else "")
                         + ("_off" if c[5] else ""))
def test_packed_operands_exact(dtype, case):
    M, N, K, apad, bpad, aoff, boff = case
    A, B = make_operands(M, N, K, dtype, "ints", seed=70)
    if apad:
        A = _padded(A, apad)
    if bpad:
        B = _padded(B, bpad)
    eb = ELEM[dtype]
    plan = tg.gemm_plan(M, N, K, tg.DTYPES[dtype], aoff * eb, A.stride(0), boff * eb, B.stride(0), 0, N).as_dict()
    if not (plan["pack_a"] or plan["pack_b"]):
        pytest.skip("both operands are TMA-addressable here")
    C = run_gemm(A, B, dtype, a_offset=aoff, b_offset=boff)
    Cref, _ = oracle_full(A, B, dtype)
    assert np.array_equal(C.astype(np.float64), Cref), f"max |diff| {np.max(np.abs(C - Cref))}"


def test_back_to_back_packed_calls_without_sync():
    """Eight calls on one stream, two ragged shapes in turn, each packing both
    operands into its own workspace from the stream-ordered pool (memory the
    previous call freed), then one check."""
    shapes = [(1000, 1001, 999), (777, 513, 1025)]
    ops = [make_operands(M, N, K, "bf16", "ints", seed=80 + i) for i, (M, N, K) in enumerate(shapes)]
    dev = [(a.cuda(), b.cuda()) for a, b in ops]
    outs = []
    s = torch.cuda.current_stream().cuda_stream
    for i in range(8):
        j = i % 2
        M, N, K = shapes[j]
        plan = tg.gemm_plan(M, N, K, tg.GEMM_BF16, 0, K, 0, N, 0, N)
        assert plan.pack_a == 1 and plan.pack_b == 1
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        a, b = dev[j]
        rc = tg.gemm_run(M, N, K, tg.GEMM_BF16, a.data_ptr(), K, b.data_ptr(), N, C.data_ptr(), N, s)
        assert rc == tg.GEMM_OK, tg.gemm_last_error()
        outs.append((j, C))
    assert tg.gemm_get_status(s) == tg.GEMM_OK, tg.gemm_last_error()
    refs = [oracle_full(a, b, "bf16")[0] for a, b in ops]
    for j, C in outs:
        assert np.array_equal(C.cpu().numpy().astype(np.float64), refs[j])

