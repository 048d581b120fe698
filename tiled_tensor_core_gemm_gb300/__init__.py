"""GB300-native dense GEMM: C = A.B over row-major operands, FP32 output, with
an optional fused epilogue C = act(alpha * A.B + beta * C + bias) stored as
FP32, BF16 or FP16.

A thin ctypes binding over the C ABI in include/gemm.h (libtcgemm.so, built
in-tree by ``build.build()``).  The functions below carry the C names and only
marshal arguments; every step of the computation runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is missing, every call
raises.

    gemm_run(M, N, K, dtype, A, lda, B, ldb, C, ldc, stream) -> status
        A, B, C are device addresses (ints); stream is a cudaStream_t as int.
    gemm_run_ex(M, N, K, dtype, A, lda, B, ldb, C, ldc, epilogue, stream) -> status
        epilogue: a GemmEpilogue (or None for plain gemm_run behaviour).
    gemm(A, B, C=None, dtype=None, stream=None) -> C
        torch-tensor convenience: row-major CUDA tensors in, FP32 C out.
    gemm_ex(A, B, C=None, alpha=1, beta=0, bias=None, act="none", out="f32", ...) -> C
        the same with the fused epilogue.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libtcgemm.so")

GEMM_FP32, GEMM_TF32, GEMM_BF16, GEMM_FP16, GEMM_E4M3, GEMM_E5M2 = 0, 1, 2, 3, 4, 5
DTYPES = {"fp32": GEMM_FP32, "tf32": GEMM_TF32, "bf16": GEMM_BF16, "fp16": GEMM_FP16, "e4m3": GEMM_E4M3,
          "e5m2": GEMM_E5M2}

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED = 2
GEMM_ERR_CUDA = 3
GEMM_ERR_TIMEOUT = 4
GEMM_ERR_NO_MEMORY = 5

GEMM_ACT_NONE, GEMM_ACT_RELU, GEMM_ACT_GELU = 0, 1, 2
ACTIVATIONS = {"none": GEMM_ACT_NONE, "relu": GEMM_ACT_RELU, "gelu": GEMM_ACT_GELU}
GEMM_OUT_F32, GEMM_OUT_BF16, GEMM_OUT_F16 = 0, 1, 2
OUT_TYPES = {"f32": GEMM_OUT_F32, "bf16": GEMM_OUT_BF16, "f16": GEMM_OUT_F16}

EXPORTED = ("gemm_run", "gemm_last_error", "gemm_get_status", "gemm_set_option",
            "gemm_get_option", "gemm_plan", "gemm_version", "gemm_run_tf32_static", "gemm_run_ex",
            "gemm_run_grouped")
TF32_STATIC_SCRATCH_BYTES = 16 * 1024 * 1024   # GEMM_TF32_STATIC_SCRATCH_BYTES in include/gemm.h


class GemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"gemm status {status}: {message}")
        self.status = status


class GemmPlan(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "path", "bm", "bn", "bk", "stages", "cta_group", "group_m", "grid", "tiles",
        "pack_a", "pack_b", "tma_store", "vec", "smem_bytes", "b_kmajor", "splits", "tail_tiles", "sched",
        "half_tiles", "cluster_split", "kb_split")]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmEpilogue(ctypes.Structure):
    """gemm_epilogue_t: y = act(alpha * acc + beta * C_old + bias[col]) stored as out_dtype."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("activation", ctypes.c_int32), ("out_dtype", ctypes.c_int32)]


class GemmGroup(ctypes.Structure):
    """gemm_group_t: one GEMM of a grouped launch (device addresses as ints)."""
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("A", ctypes.c_void_p),
                ("lda", ctypes.c_int64), ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("C", ctypes.c_void_p),
                ("ldc", ctypes.c_int64), ("bias", ctypes.c_void_p)]


def make_epilogue(alpha=1.0, beta=0.0, bias=0, act="none", out="f32") -> GemmEpilogue:
    """A GemmEpilogue from names; bias is a device address (0 for none)."""
    return GemmEpilogue(float(alpha), float(beta), int(bias) or None, ACTIVATIONS[act], OUT_TYPES[out])


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load libtcgemm.so; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with tiled_tensor_core_gemm_gb300.build.build() "
                               "(there is no fallback path)")
        lib = ctypes.CDLL(LIB_PATH)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.gemm_run.argtypes = [i64, i64, i64, ctypes.c_int, p, i64, p, i64, p, i64, p]
        lib.gemm_run.restype = ctypes.c_int
        lib.gemm_last_error.argtypes = []
        lib.gemm_last_error.restype = ctypes.c_char_p
        lib.gemm_get_status.argtypes = [p]
        lib.gemm_get_status.restype = ctypes.c_int
        lib.gemm_set_option.argtypes = [ctypes.c_char_p, i64]
        lib.gemm_set_option.restype = ctypes.c_int
        lib.gemm_get_option.argtypes = [ctypes.c_char_p]
        lib.gemm_get_option.restype = i64
        lib.gemm_plan.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_uint64, i64, ctypes.c_uint64, i64,
                                  ctypes.c_uint64, i64, ctypes.c_int32, ctypes.POINTER(GemmPlan)]
        lib.gemm_plan.restype = ctypes.c_int
        lib.gemm_version.argtypes = []
        lib.gemm_version.restype = ctypes.c_int
        lib.gemm_run_tf32_static.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, p]
        lib.gemm_run_tf32_static.restype = ctypes.c_int
        lib.gemm_run_ex.argtypes = [i64, i64, i64, ctypes.c_int, p, i64, p, i64, p, i64, ctypes.POINTER(GemmEpilogue),
                                    p]
        lib.gemm_run_ex.restype = ctypes.c_int
        lib.gemm_run_grouped.argtypes = [ctypes.c_int, i64, ctypes.POINTER(GemmGroup), ctypes.POINTER(GemmEpilogue), p]
        lib.gemm_run_grouped.restype = ctypes.c_int
        _lib = lib
        return lib


# ------------------------------------------------------------ C-ABI mirrors ---
def gemm_run(M, N, K, dtype, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return load_library().gemm_run(M, N, K, dtype, A, lda, B, ldb, C, ldc, stream)


def gemm_last_error() -> str:
    return load_library().gemm_last_error().decode()


def gemm_get_status(stream=0) -> int:
    return load_library().gemm_get_status(stream)


def gemm_set_option(key: str, value: int) -> int:
    return load_library().gemm_set_option(key.encode(), int(value))


def gemm_get_option(key: str) -> int:
    return int(load_library().gemm_get_option(key.encode()))


def gemm_plan(M, N, K, dtype, a_addr, lda, b_addr, ldb, c_addr, ldc, num_sms=0) -> GemmPlan:
    out = GemmPlan()
    rc = load_library().gemm_plan(M, N, K, dtype, a_addr, lda, b_addr, ldb, c_addr, ldc, num_sms,
                                  ctypes.byref(out))
    if rc != GEMM_OK:
        raise GemmError(rc, gemm_last_error())
    return out


def gemm_version() -> int:
    return load_library().gemm_version()


def gemm_run_tf32_static(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """TF32 C = A.B that allocates no device memory (scratch in a fixed library array)."""
    return load_library().gemm_run_tf32_static(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_run_ex(M, N, K, dtype, A, lda, B, ldb, C, ldc, epilogue=None, stream=0) -> int:
    """C = act(alpha * A.B + beta * C + bias) stored as the epilogue's output type."""
    ep = ctypes.byref(epilogue) if epilogue is not None else None
    return load_library().gemm_run_ex(M, N, K, dtype, A, lda, B, ldb, C, ldc, ep, stream)


def gemm_run_grouped(dtype, groups, epilogue=None, stream=0) -> int:
    """A batch of independent GEMMs in one launch; groups: a sequence of GemmGroup."""
    arr = (GemmGroup * len(groups))(*groups) if len(groups) else None
    ep = ctypes.byref(epilogue) if epilogue is not None else None
    return load_library().gemm_run_grouped(dtype, len(groups), arr, ep, stream)


# ------------------------------------------------------ tensor convenience ---
def _ld(t) -> int:
    if t.dim() != 2:
        raise ValueError("operands must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("operands must be row-major (unit stride along columns)")
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def _same_cuda_device(*tensors):
    """Every tensor given (None entries skipped) is a CUDA tensor on one device."""
    live = [t for t in tensors if t is not None]
    for t in live:
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors (this library has no CPU path)")
        if t.device != live[0].device:
            raise ValueError(f"tensors on different devices: {live[0].device} and {t.device}")


def _check_bias(torch, bias, n):
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != n or not bias.is_contiguous()):
        raise TypeError(f"bias must be {n} contiguous float32 values")


def _operand_types(torch):
    """dtype code -> torch element type of A and B."""
    return {GEMM_BF16: torch.bfloat16, GEMM_FP16: torch.float16, GEMM_E4M3: torch.float8_e4m3fn,
            GEMM_E5M2: torch.float8_e5m2}


def _default_dtype(torch, t) -> str:
    return {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float8_e4m3fn: "e4m3",
            torch.float8_e5m2: "e5m2"}.get(t.dtype, "fp32")


def gemm(A, B, C=None, dtype=None, stream=None):
    """C = A.B through gemm_run for CUDA tensors (float32, bfloat16, float16 or float8).

    dtype: "fp32" (default for float32 inputs), "tf32", "bf16", "fp16", "e4m3"
    or "e5m2" (the defaults for bfloat16, float16, float8_e4m3fn and
    float8_e5m2 inputs).  C, if given, must be a float32 CUDA tensor of shape
    (M, N); it is overwritten.
    """
    import torch

    if dtype is None:
        dtype = _default_dtype(torch, A)
    code = DTYPES[dtype]
    want = _operand_types(torch).get(code, torch.float32)
    if A.dtype != want or B.dtype != want:
        raise TypeError(f"{dtype} GEMM takes {want} operands")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if C is not None and (C.dtype != torch.float32 or tuple(C.shape) != (M, N)):
        raise TypeError(f"C must be a ({M}, {N}) float32 tensor")
    _same_cuda_device(A, B, C)
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    rc = gemm_run(M, N, K, code, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C), stream)
    if rc != GEMM_OK:
        raise GemmError(rc, gemm_last_error())
    return C


def gemm_ex(A, B, C=None, alpha=1.0, beta=0.0, bias=None, act="none", out="f32", dtype=None, stream=None):
    """C = act(alpha * A.B + beta * C + bias) through gemm_run_ex for CUDA tensors.

    out: "f32", "bf16" or "f16", the element type of C (allocated if None;
    beta must then be 0).  bias: a float32 CUDA tensor of N values or None.
    """
    import torch

    if dtype is None:
        dtype = _default_dtype(torch, A)
    code = DTYPES[dtype]
    want = _operand_types(torch).get(code, torch.float32)
    if A.dtype != want or B.dtype != want:
        raise TypeError(f"{dtype} GEMM takes {want} operands")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    cdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out]
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=cdt, device=A.device)
    elif C.dtype != cdt or tuple(C.shape) != (M, N):
        raise TypeError(f"C must be a ({M}, {N}) {cdt} tensor")
    _check_bias(torch, bias, N)
    _same_cuda_device(A, B, C, bias)
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    ep = make_epilogue(alpha, beta, bias.data_ptr() if bias is not None else 0, act, out)
    rc = gemm_run_ex(M, N, K, code, A.data_ptr(), _ld(A), B.data_ptr(), _ld(B), C.data_ptr(), _ld(C), ep, stream)
    if rc != GEMM_OK:
        raise GemmError(rc, gemm_last_error())
    return C


def gemm_grouped(As, Bs, Cs=None, biases=None, alpha=1.0, beta=0.0, act="none", out="f32", dtype=None, stream=None):
    """C_g = act(alpha * A_g.B_g + beta * C_g + bias_g) for every g, in one grouped launch.

    As, Bs: sequences of row-major CUDA tensors of one type; Cs (allocated if
    None, beta must then be 0) in the output type; biases: None or a sequence
    of float32 tensors of N_g values (or None entries).  Returns the Cs.
    """
    import torch

    if len(As) != len(Bs) or (Cs is not None and len(Cs) != len(As)) or (biases is not None and len(biases) != len(As)):
        raise ValueError("As, Bs, Cs and biases differ in length")
    if not As:
        return []
    if dtype is None:
        dtype = _default_dtype(torch, As[0])
    code = DTYPES[dtype]
    want = _operand_types(torch).get(code, torch.float32)
    cdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out]
    if Cs is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs Cs")
        Cs = [torch.empty((a.shape[0], b.shape[1]), dtype=cdt, device=a.device) for a, b in zip(As, Bs)]
    groups = []
    for i, (a, b, c) in enumerate(zip(As, Bs, Cs)):
        if a.dtype != want or b.dtype != want:
            raise TypeError(f"{dtype} GEMM takes {want} operands")
        if a.shape[1] != b.shape[0] or tuple(c.shape) != (a.shape[0], b.shape[1]) or c.dtype != cdt:
            raise ValueError(f"group {i}: shapes or C type do not match")
        bias = biases[i] if biases is not None else None
        _check_bias(torch, bias, b.shape[1])
        _same_cuda_device(As[0], a, b, c, bias)
        groups.append(GemmGroup(a.shape[0], b.shape[1], a.shape[1], a.data_ptr(), _ld(a), b.data_ptr(), _ld(b),
                                c.data_ptr(), _ld(c), bias.data_ptr() if bias is not None else None))
    if stream is None:
        stream = torch.cuda.current_stream(As[0].device).cuda_stream
    ep = make_epilogue(alpha, beta, 0, act, out)
    rc = gemm_run_grouped(code, groups, ep, stream)
    if rc != GEMM_OK:
        raise GemmError(rc, gemm_last_error())
    return Cs
