"""Helpers for the GPU parity tests: run the library through its C ABI on
seeded inputs and compare with the oracle.

Acceptance metric: r = max_ij |C_ij - Cref_ij| / D_ij with D = |A|.|B| (fp64);
D_ij == 0 requires C_ij == Cref_ij exactly; any NaN/Inf fails.  Bounds: 1e-5
for FP32 and for BF16, FP16 or FP8 inputs with FP32 accumulation (the oracle
uses the rounded narrow inputs, whose products are exact in FP32, so only the
accumulation error counts), 2e-3 for TF32.
Derivation of the TF32 bound: the tensor cores read each FP32 operand with a
10-bit mantissa; whether they round or truncate, each operand's relative
error is below 2^-10, so each product's is below (1 + 2^-10)^2 - 1 < 1.96e-3,
and sum_k |err_k| <= 1.96e-3 * D; FP32 accumulation adds about K * 2^-24 * D
at worst, which keeps r under 2e-3 for K <= 8192.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tiled_tensor_core_gemm_gb300 as tg
from tiled_tensor_core_gemm_gb300.inputs import as_oracle_array

TOL = {"fp32": 1e-5, "bf16": 1e-5, "fp16": 1e-5, "tf32": 2e-3, "e4m3": 1e-5, "e5m2": 1e-5}
FP8 = ("e4m3", "e5m2")
GUARD = 256   # NaN-filled floats before and after C


def to_device(x: torch.Tensor, offset_elems: int = 0):
    """Copy a (possibly padded) CPU operand to the GPU keeping its leading
    dimension; optionally start it `offset_elems` elements into its buffer.
    Returns (keepalive tensor, device address, leading dimension)."""
    rows, cols = x.shape
    ld = x.stride(0) if rows > 1 else max(cols, 1)
    if rows == 0 or cols == 0:
        buf = torch.empty(max(offset_elems, 1) + 1, dtype=x.dtype, device="cuda")
        return buf, buf.data_ptr() + offset_elems * x.element_size(), ld
    flat = torch.as_strided(x, (rows, ld), (ld, 1)) if ld != cols else x
    buf = torch.empty(offset_elems + rows * ld, dtype=x.dtype, device="cuda")
    buf[offset_elems:].copy_(flat.reshape(-1).contiguous())
    return buf, buf.data_ptr() + offset_elems * x.element_size(), ld


def run_gemm(A: torch.Tensor, B: torch.Tensor, dtype: str, ldc_pad: int = 0, a_offset: int = 0,
             b_offset: int = 0, stream=None) -> np.ndarray:
    """C = A.B on the GPU via gemm_run; checks the status word and that nothing
    outside C (guard bands, ldc padding) was written.  Returns C as float32."""
    M, K = A.shape
    N = B.shape[1]
    a_keep, a_ptr, lda = to_device(A, a_offset)
    b_keep, b_ptr, ldb = to_device(B, b_offset)
    ldc = max(N, 1) + ldc_pad
    cbuf = torch.full((2 * GUARD + M * ldc,), float("nan"), dtype=torch.float32, device="cuda")
    c_ptr = cbuf.data_ptr() + GUARD * 4
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    rc = tg.gemm_run(M, N, K, tg.DTYPES[dtype], a_ptr, lda, b_ptr, ldb, c_ptr, ldc, stream)
    assert rc == tg.GEMM_OK, tg.gemm_last_error()
    st = tg.gemm_get_status(stream)
    assert st == tg.GEMM_OK, tg.gemm_last_error()
    host = cbuf.cpu().numpy()
    del a_keep, b_keep
    assert np.all(np.isnan(host[:GUARD])), "write before C"
    assert np.all(np.isnan(host[GUARD + M * ldc:])), "write after C"
    C = host[GUARD:GUARD + M * ldc].reshape(M, ldc)
    if ldc_pad:
        assert np.all(np.isnan(C[:, N:])), "write into the ldc padding"
    return C[:, :N].copy()


def tf32_round(x: np.ndarray, mode: str) -> np.ndarray:
    """FP32 values cut to TF32's 10 mantissa bits, as FP32: "rz" drops the
    13 low bits (toward zero), "rn" rounds to the nearest TF32 value with
    ties to an even last bit.  The pages give only the format (FP32 range,
    10-bit mantissa), not how the tensor cores reduce an FP32 operand to it;
    the two diagnostic oracles built from these inputs tell which one a
    kernel's output follows.  Finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    if mode == "rz":
        r = u & np.uint32(0xFFFFE000)
    elif mode == "rn":
        # add just under half of the dropped part's range, plus the kept last bit
        # (so an exact half rounds to even), then drop; a carry moves into the
        # exponent as it should, and the sign bit is untouched
        r = (u + np.uint32(0x0FFF) + ((u >> np.uint32(13)) & np.uint32(1))) & np.uint32(0xFFFFE000)
    else:
        raise ValueError(f"unknown rounding mode {mode!r}")
    return r.view(np.float32)


def error_ratio(C: np.ndarray, Cref: np.ndarray, D: np.ndarray) -> float:
    C = C.astype(np.float64)
    if not np.all(np.isfinite(C)):
        return float("inf")
    diff = np.abs(C - Cref)
    zero = D == 0
    if np.any(diff[zero] != 0):
        return float("inf")
    if not np.any(~zero):
        return 0.0
    return float(np.max(diff[~zero] / D[~zero]))


def oracle_full(A: torch.Tensor, B: torch.Tensor, dtype: str):
    return oracle.gemm(as_oracle_array(A), as_oracle_array(B), bf16=(dtype == "bf16"), fp16=(dtype == "fp16"),
                       fp8=dtype if dtype in FP8 else None, with_scale=True)


def oracle_rows(A: torch.Tensor, B: torch.Tensor, dtype: str, rows):
    return oracle.gemm_rows(as_oracle_array(A), as_oracle_array(B), rows, bf16=(dtype == "bf16"),
                            fp16=(dtype == "fp16"), fp8=dtype if dtype in FP8 else None)


def sample_rows(M: int, tile: int = 128, extra: int = 8, seed: int = 0):
    """Rows at every 8th tile boundary (first and last row of the tile), the
    last rows of the matrix, and a few seeded random rows."""
    rows = set()
    for t in range(0, M, tile * 8):
        rows.update({t, min(t + tile - 1, M - 1)})
    rows.update({0, M - 1, max(M - 2, 0)})
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, M, extra))
    return sorted(rows)


# ----------------------------------------------------------- fused epilogue --
# Acceptance for C = act(alpha * A.B + beta * C_old + bias) stored as `out`:
# the stored value must lie in [RN(y - b), RN(y + b)], RN being round to
# nearest (ties to even) onto the output type's grid, y the oracle's fp64
# value and b a bound on the error of the FP32 result before the cast:
#   b = (1.13 * tol + 1e-6) * S,  S = |alpha| D + |beta C_old| + |bias|,
# i.e. the GEMM's own bound on alpha * A.B, times the largest slope of the
# activation (GELU's is below 1.13, ReLU's is 1), plus a few FP32 roundings of
# the three-term sum and of the activation.  A round-to-nearest cast is
# monotone, so the cast of any FP32 value within b of y lands in that
# interval; where b is small against the output's spacing the interval is the
# single grid point RN(y), and a cast that rounds up, truncates or lands one
# grid step away falls outside it.
OUT_P = {"f32": 24, "bf16": 8, "f16": 11}          # significand bits
OUT_EMIN = {"f32": -126, "bf16": -126, "f16": -14}  # smallest normal exponent


def grid_round(x: np.ndarray, out: str, up: bool) -> np.ndarray:
    """x rounded down (up=False) or up to the output type's representable grid."""
    x = np.asarray(x, np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e - 1, OUT_EMIN[out])
    ulp = np.ldexp(1.0, e - (OUT_P[out] - 1))
    q = x / ulp
    return (np.ceil(q) if up else np.floor(q)) * ulp


def grid_round_nearest(x: np.ndarray, out: str) -> np.ndarray:
    """x rounded to the nearest point of the output type's grid, ties to the
    point with an even last significand bit (values in the type's range)."""
    x = np.asarray(x, np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e - 1, OUT_EMIN[out])
    ulp = np.ldexp(1.0, e - (OUT_P[out] - 1))
    return np.rint(x / ulp) * ulp


OUT_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def run_gemm_ex(A: torch.Tensor, B: torch.Tensor, dtype: str, out: str = "f32", alpha: float = 1.0,
                beta: float = 0.0, c_old: torch.Tensor | None = None, bias: torch.Tensor | None = None,
                act: str = "none", ldc_pad: int = 0, epilogue: bool = True) -> np.ndarray:
    """C through gemm_run_ex on the GPU (C starts as c_old when given); checks the
    status word and that nothing outside C (guard bands, ldc padding) was
    written.  Returns C as float64.  epilogue=False passes a NULL epilogue."""
    M, K = A.shape
    N = B.shape[1]
    a_keep, a_ptr, lda = to_device(A)
    b_keep, b_ptr, ldb = to_device(B)
    ldc = max(N, 1) + ldc_pad
    cdt = OUT_TORCH[out]
    cbuf = torch.full((2 * GUARD + M * ldc,), float("nan"), dtype=cdt, device="cuda")
    body = cbuf[GUARD:GUARD + M * ldc].view(M, ldc) if M * ldc else None
    if c_old is not None and M and N:
        body[:, :N].copy_(c_old.to(cdt))
    c_ptr = cbuf.data_ptr() + GUARD * cbuf.element_size()
    bias_d = bias.to(torch.float32).contiguous().cuda() if bias is not None else None
    stream = torch.cuda.current_stream().cuda_stream
    ep = tg.make_epilogue(alpha, beta, bias_d.data_ptr() if bias_d is not None else 0, act, out) if epilogue else None
    rc = tg.gemm_run_ex(M, N, K, tg.DTYPES[dtype], a_ptr, lda, b_ptr, ldb, c_ptr, ldc, ep, stream)
    assert rc == tg.GEMM_OK, tg.gemm_last_error()
    st = tg.gemm_get_status(stream)
    assert st == tg.GEMM_OK, tg.gemm_last_error()
    host = cbuf.cpu().to(torch.float64).numpy()
    del a_keep, b_keep
    assert np.all(np.isnan(host[:GUARD])), "write before C"
    assert np.all(np.isnan(host[GUARD + M * ldc:])), "write after C"
    C = host[GUARD:GUARD + M * ldc].reshape(M, ldc)
    if ldc_pad:
        assert np.all(np.isnan(C[:, N:])), "write into the ldc padding"
    return C[:, :N].copy()


def oracle_c_old(c_old: torch.Tensor | None, out: str):
    """The old C as the oracle takes it (float32 or 16-bit patterns)."""
    if c_old is None:
        return None
    return as_oracle_array(c_old.to(OUT_TORCH[out])).copy()


def epilogue_check(C: np.ndarray, acc: np.ndarray, D: np.ndarray, dtype: str, out: str, alpha: float, beta: float,
                   c_old, bias, act: str):
    """Worst |out - mid| / half over the elements, where [lo, hi] = [RN(y - b),
    RN(y + b)] is the allowed interval, mid its centre and half its half
    width; <= 1 passes (inside the interval), and an element whose interval is
    a single grid point must equal it (else inf).  Also returns y."""
    old = oracle_c_old(c_old, out)
    b = bias.numpy() if bias is not None else None
    y = oracle.epilogue(acc, alpha, beta, old, out, b, act)
    S = abs(alpha) * D
    if beta != 0.0:
        S = S + abs(beta) * np.abs(oracle.epilogue(np.zeros_like(acc), 0.0, 1.0, old, out))
    if b is not None:
        S = S + np.abs(b.astype(np.float64))[None, :]
    slack = (1.13 * TOL[dtype] + 1e-6) * S
    lo = grid_round_nearest(y - slack, out)
    hi = grid_round_nearest(y + slack, out)
    if not np.all(np.isfinite(C)):
        return float("inf"), y
    mid, half = (lo + hi) / 2, (hi - lo) / 2
    diff = np.abs(C - mid)
    point = half == 0
    if np.any(diff[point] != 0):
        return float("inf"), y
    live = ~point
    return (float(np.max(diff[live] / half[live])) if np.any(live) else 0.0), y
