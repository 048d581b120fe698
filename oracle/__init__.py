"""Dense GEMM oracle (test infrastructure only).

A plain, slow, obviously correct C = A.B in double precision, compiled from
``gemm_oracle.c`` with gcc and reached through ctypes.  Only ``tests/``, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import this package; the product library never does, and this package imports
nothing from it.

What it computes: "Shared memory and tensor cores" (ml-compiler-from-scratch
ch. 13) section 13.1 defines the GEMM as C = A @ B with 2*M*N*K flops; section
13.8 fixes that tensor-core products are exact and sums are FP32.  The oracle
forms the same exact products and sums them in fp64 (k ascending), so it is at
least as accurate as any path under test.  BF16 and FP16 inputs are passed as
their raw 16-bit patterns, FP8 (E4M3, E5M2) inputs as bytes; all are widened
exactly.

``epilogue`` applies the fused epilogue of section 13.10 (bias, activation,
residual add, output type) to an fp64 product: y = act(alpha * acc + beta *
c_old + bias[j]), returned unrounded.

Every GEMM function also returns D[i, j] = sum_k |A[i, k]| * |B[k, j]| on request,
the per-entry scale used by the acceptance test max|C - C_ref| / D.

Pins (tests/test_oracle.py): identity and permutation products, all-ones inputs
(C == K everywhere), small-integer inputs against exact integer arithmetic, a
second independent loop order at tiny sizes, float64 library matmul, and the
BF16, FP16 and FP8 widenings against the library's own conversions; the epilogue
against the library's addmm, ReLU and GELU, printed values of the normal CDF,
GELU's odd-part identity, and per-column bias broadcasting.
tests/test_oracle_mutants.py plants one plausible mistake at a time in a copy
of gemm_oracle.c and checks that some pin fails on each.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgemm_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def compile_library(src: str, out: str) -> str:
    """Compile one C source of the oracle's form into the shared library `out`
    (gcc, OpenMP, no -march flags, so x86 and Arm hosts give the same bits)."""
    os.makedirs(os.path.dirname(os.path.abspath(out)), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
           "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle shared library."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        return compile_library(_SRC, _LIB_PATH)


def bind(path: str):
    """Load a library built by compile_library and declare its entry points.
    The module's functions use the library `_load` returns; the mutation
    tests bind a copy of the source with one planted mistake the same way."""
    lib = ctypes.CDLL(os.path.abspath(path))
    full = [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64]
    rows = [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr, _ptr]
    jik = [_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64]
    kinds = ("f32", "bf16", "f16", "e4m3", "e5m2")
    table = [(f"oracle_gemm_{k}", full) for k in kinds] + [(f"oracle_gemm_rows_{k}", rows) for k in kinds]
    table += [(f"oracle_gemm_{k}_jik", jik) for k in kinds]
    table += [(f"oracle_widen_{k}", [_ptr, _ptr, _i64]) for k in ("bf16", "f16", "e4m3", "e5m2")]
    for name, args in table:
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = None
    lib.oracle_epilogue.argtypes = [_i64, _i64, _ptr, _i64, ctypes.c_double, ctypes.c_double, _ptr,
                                    ctypes.c_int, _i64, _ptr, ctypes.c_int, _ptr, _i64]
    lib.oracle_epilogue.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


def num_threads() -> int:
    """Host threads the oracle's OpenMP loops use."""
    return int(_load().oracle_num_threads())


_STORAGE = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16, "e4m3": np.uint8, "e5m2": np.uint8}


def _as_operand(x: np.ndarray, kind: str) -> np.ndarray:
    want = _STORAGE[kind]
    if x.dtype != want:
        raise TypeError(f"oracle operand must be {want.__name__}, got {x.dtype}")
    if x.ndim != 2 or (x.size > 0 and x.shape[1] > 1 and x.strides[1] != x.itemsize):
        raise ValueError("oracle operands are row-major 2-D arrays with unit inner stride")
    return x


def _ld(x: np.ndarray) -> int:
    return x.strides[0] // x.itemsize if (x.shape[0] > 1 and x.size > 0) else max(x.shape[1], 1)


def _kind(bf16: bool, fp16: bool, fp8=None) -> str:
    if (bf16, fp16, fp8 is not None).count(True) > 1:
        raise ValueError("bf16, fp16 and fp8 are exclusive")
    if fp8 is not None:
        if fp8 not in ("e4m3", "e5m2"):
            raise ValueError(f"unknown FP8 format {fp8!r}")
        return fp8
    return "bf16" if bf16 else "f16" if fp16 else "f32"


def gemm(A: np.ndarray, B: np.ndarray, bf16: bool = False, with_scale: bool = False, fp16: bool = False,
         fp8=None):
    """C = A.B in fp64 (and D = |A|.|B| if with_scale).

    A: M x K, B: K x N, row-major, float32, or uint16 patterns of BF16
    (bf16=True) or IEEE half (fp16=True), or uint8 patterns of an FP8 format
    (fp8="e4m3" or "e5m2").
    """
    kind = _kind(bf16, fp16, fp8)
    _as_operand(A, kind), _as_operand(B, kind)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    C = np.empty((M, N), np.float64)
    D = np.empty((M, N), np.float64) if with_scale else None
    fn = getattr(_load(), f"oracle_gemm_{kind}")
    fn(M, N, K, A.ctypes.data, _ld(A), B.ctypes.data, _ld(B), C.ctypes.data, max(N, 1),
       D.ctypes.data if D is not None else None, max(N, 1))
    return (C, D) if with_scale else C


def gemm_rows(A: np.ndarray, B: np.ndarray, rows, bf16: bool = False, with_scale: bool = True, fp16: bool = False,
              fp8=None):
    """Rows `rows` of C = A.B and (with_scale) of D = |A|.|B|, each len(rows) x N, fp64."""
    kind = _kind(bf16, fp16, fp8)
    _as_operand(A, kind), _as_operand(B, kind)
    M, K = A.shape
    N = B.shape[1]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= M):
        raise IndexError("row index out of range")
    C = np.empty((r.size, N), np.float64)
    D = np.empty((r.size, N), np.float64) if with_scale else None
    fn = getattr(_load(), f"oracle_gemm_rows_{kind}")
    fn(M, N, K, A.ctypes.data, _ld(A), B.ctypes.data, _ld(B), r.ctypes.data, r.size,
       C.ctypes.data, D.ctypes.data if D is not None else None)
    return C, D


def gemm_jik(A: np.ndarray, B: np.ndarray, bf16: bool = False, fp16: bool = False, fp8=None) -> np.ndarray:
    """The same product with the j-i-k loop order (tiny sizes only)."""
    kind = _kind(bf16, fp16, fp8)
    _as_operand(A, kind), _as_operand(B, kind)
    M, K = A.shape
    N = B.shape[1]
    C = np.empty((M, N), np.float64)
    fn = getattr(_load(), f"oracle_gemm_{kind}_jik")
    fn(M, N, K, A.ctypes.data, _ld(A), B.ctypes.data, _ld(B), C.ctypes.data, max(N, 1))
    return C


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact value of each BF16 pattern, as fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_widen_bf16(b.ctypes.data, out.ctypes.data, b.size)
    return out


def widen_f16(bits: np.ndarray) -> np.ndarray:
    """Exact value of each IEEE half pattern, as fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_widen_f16(b.ctypes.data, out.ctypes.data, b.size)
    return out


def widen_fp8(bits: np.ndarray, fmt: str) -> np.ndarray:
    """Exact value of each FP8 byte (fmt "e4m3" or "e5m2"), as fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(b.shape, np.float64)
    getattr(_load(), f"oracle_widen_{_kind(False, False, fmt)}")(b.ctypes.data, out.ctypes.data, b.size)
    return out


ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2}
OUT_TYPES = {"f32": 0, "bf16": 1, "f16": 2}


def epilogue(acc: np.ndarray, alpha: float = 1.0, beta: float = 0.0, c_old=None, out: str = "f32",
             bias=None, act: str = "none") -> np.ndarray:
    """y = act(alpha * acc + beta * c_old + bias[j]) in fp64, unrounded.

    acc: M x N fp64 product.  c_old: M x N C already in memory, float32 for
    out="f32" or the uint16 patterns of BF16 / IEEE half; read only when
    beta != 0.  bias: N float32 values or None.  act: "none", "relu", "gelu".
    """
    a = np.ascontiguousarray(acc, dtype=np.float64)
    if a.ndim != 2:
        raise ValueError("acc must be 2-D")
    M, N = a.shape
    if out not in OUT_TYPES or act not in ACTIVATIONS:
        raise ValueError(f"unknown output type {out!r} or activation {act!r}")
    old = None
    if beta != 0.0:
        if c_old is None:
            raise ValueError("beta != 0 needs c_old")
        old = np.ascontiguousarray(c_old, dtype=np.float32 if out == "f32" else np.uint16)
        if old.shape != (M, N):
            raise ValueError("c_old must match acc")
    b = None
    if bias is not None:
        b = np.ascontiguousarray(bias, dtype=np.float32)
        if b.shape != (N,):
            raise ValueError("bias must hold N values")
    Y = np.empty((M, N), np.float64)
    _load().oracle_epilogue(M, N, a.ctypes.data, max(N, 1), float(alpha), float(beta),
                            old.ctypes.data if old is not None else None, OUT_TYPES[out], max(N, 1),
                            b.ctypes.data if b is not None else None, ACTIVATIONS[act], Y.ctypes.data, max(N, 1))
    return Y
