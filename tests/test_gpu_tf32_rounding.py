"""Which TF32 reading of FP32 operands the tensor cores follow (a diagnostic,
not the acceptance test, which compares with the unrounded FP32 inputs).

The pages fix TF32 as FP32's range with a 10-bit mantissa but not how an FP32
operand is cut to it.  Two diagnostic oracles take the inputs pre-rounded to
TF32, toward zero (RZ) and to nearest-even (RN); the kernel's output follows
the one whose residual is only FP32 accumulation error (about 1e-7 of D),
while the other leaves the rounding difference itself (about 1e-4).  The
inputs carry random low mantissa bits, so the two readings differ on most
elements."""
import numpy as np
import pytest

import oracle
import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300 import build as tgbuild
from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array, make_operands

from gemm_check import TOL, error_ratio, run_gemm, tf32_round

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    tgbuild.build()
    tg.load_library()
    yield


@pytest.mark.parametrize("M,N,K", [(512, 384, 1024), (300, 260, 333)])
def test_tf32_operands_are_read_toward_zero(M, N, K):
    A, B = make_operands(M, N, K, "tf32", "normal", seed=140)
    C = run_gemm(A, B, "tf32").astype(np.float64)
    a, b = as_oracle_array(A), as_oracle_array(B)
    ref, D = oracle.gemm(a, b, with_scale=True)
    r = {"fp32": error_ratio(C, ref, D)}
    for mode in ("rz", "rn"):
        ref_m = oracle.gemm(tf32_round(a, mode), tf32_round(b, mode))
        r[mode] = error_ratio(C, ref_m, D)
    print(f"TF32 {M}x{N}x{K}: r against unrounded inputs {r['fp32']:.2e}, "
          f"RZ-rounded {r['rz']:.2e}, RN-rounded {r['rn']:.2e}")
    assert r["fp32"] <= TOL["tf32"]
    assert r["rz"] <= 1e-5 < r["rn"], r
