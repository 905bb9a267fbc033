"""GB300-native (sm_103a) single-precision GEMM: C = alpha*A*B + beta*C.

The computation runs entirely in the CUDA library ``libsgemm_gb300.so``
(C ABI in ``include/sgemm_gb300.h``).  This module only marshals arguments
to that ABI through ctypes: the functions named like the C entry points take
the same arguments (device pointers as integers, streams as handles), and
``matmul`` adapts torch CUDA tensors to them.  There is no CPU fallback: if
the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import _build_ext

__all__ = [
    "SGEMM_ALGO_AUTO", "SGEMM_ALGO_FFMA", "SGEMM_ALGO_TF32X3",
    "SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE", "SGEMM_FLAG_TILE_ROWS", "SGEMM_FLAG_WHOLE_TILES", "SGEMM_FLAG_SPLIT_TAIL",
    "SGEMM_FLAG_PAIRS", "SGEMM_FLAG_NO_PAIRS",
    "SGEMM_ERR_DEVICE_TIMEOUT",
    "SgemmError", "library", "lib_path", "declared_functions",
    "sgemm", "sgemm_ex", "sgemm_host", "sgemm_host_blocks", "sgemm_plan_info", "sgemm_check_status",
    "sgemm_status_string", "sgemm_release", "sgemm_version", "sgemm_noalloc", "sgemm_noalloc_debug_flags", "sgemm_tf32_mma_rate", "sgemm_ffma_rate", "sgemm_t", "sgemm_strided_batched", "sgemm_conv2d", "sgemm_conv2d_ex", "SGEMM_CONV_NO_PAD_COPY", "conv2d_out_size", "matmul",
    "SGEMM_ERR_SCRATCH_LIMIT", "SGEMM_ERR_OUT_OF_BOUNDS",
]

SGEMM_ALGO_AUTO = 0
SGEMM_ALGO_FFMA = 1
SGEMM_ALGO_TF32X3 = 2
SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE = 1
SGEMM_FLAG_WHOLE_TILES = 2
SGEMM_FLAG_SPLIT_TAIL = 4


def SGEMM_FLAG_TILE_ROWS(r: int) -> int:
    """Force r C rows per 3xTF32 tile (16, 32, 64, 128, 192 or 256)."""
    return ((r // 16) & 0xFF) << 8


SGEMM_ERR_DEVICE_TIMEOUT = 10001
SGEMM_ERR_NO_DEVICE = 10002
SGEMM_ERR_UNSUPPORTED_DEVICE = 10003
SGEMM_ERR_WORKSPACE = 10004
SGEMM_ERR_INTERNAL = 10005
SGEMM_ERR_SCRATCH_LIMIT = 10006
SGEMM_ERR_OUT_OF_BOUNDS = 10007

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "sgemm_gb300.h")

_lock = threading.Lock()
_lib = None

_i, _f, _p = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
_SIGS = {
    "sgemm": (_i, [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p]),
    "sgemm_ex": (_i, [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p, _i, _i, _i]),
    "sgemm_host": (_i, [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _i]),
    "sgemm_plan_info": (_i, [_i, _i, _i, _p, _i, _p, _i, _p, _i, _i, _i, _i, _f, _f, _i,
                             ctypes.POINTER(ctypes.c_int), _i]),
    "sgemm_host_blocks": (_i, [_i, _i, _i, _i, _i, _i, _f, _f, _i, _i, ctypes.POINTER(ctypes.c_int),
                               ctypes.POINTER(ctypes.c_int), _i]),
    "sgemm_check_status": (_i, [_p]),
    "sgemm_status_string": (ctypes.c_char_p, [_i]),
    "sgemm_release": (_i, []),
    "sgemm_version": (_i, []),
    "sgemm_tf32_mma_rate": (_i, [_i, _i, _p, ctypes.POINTER(ctypes.c_double)]),
    "sgemm_ffma_rate": (_i, [_i, _i, _p, ctypes.POINTER(ctypes.c_double)]),
    "sgemm_t": (_i, [_i, _i, _i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p, _i]),
    "sgemm_strided_batched": (_i, [_i, _i, _i, _i, _i, _f, _p, _i, ctypes.c_longlong, _p, _i, ctypes.c_longlong,
                                   _f, _p, _i, ctypes.c_longlong, _i, _p, _i]),
    "sgemm_noalloc": (_i, [_i, _i, _i, _f, _p, _i, _p, _i, _f, _p, _i, _p, _i]),
    "sgemm_noalloc_debug_flags": (_i, [_i]),
    "sgemm_conv2d": (_i, [_i] * 13 + [_f, _p, _p, _f, _p, _p, _i]),
    "sgemm_conv2d_ex": (_i, [_i] * 13 + [_f, _p, _p, _f, _p, _p, _i, _i]),
}


class SgemmError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} returned {status}: {sgemm_status_string(status)}")


def lib_path() -> str:
    return _build_ext.lib_path()


def declared_functions() -> list[str]:
    """Names of the functions declared in the C header."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sgemm\w*)\s*\(", text, flags=re.M)


def library() -> ctypes.CDLL:
    """Load the CUDA library (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library not built: {path} is missing; run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def _stream(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return int(getattr(stream, "cuda_stream"))  # torch.cuda.Stream


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


# ------------------------------------------------------- C ABI, same names

def sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    return library().sgemm(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                           _stream(stream))


def sgemm_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, algo=0, splits=0,
             flags=0) -> int:
    return library().sgemm_ex(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                              _stream(stream), algo, splits, flags)


def sgemm_t(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, algo=0) -> int:
    return library().sgemm_t(int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                             _ptr(C), ldc, _stream(stream), algo)


def sgemm_strided_batched(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                          strideC, batch, stream=None, algo=0) -> int:
    return library().sgemm_strided_batched(int(transa), int(transb), M, N, K, alpha, _ptr(A), lda, strideA,
                                           _ptr(B), ldb, strideB, beta, _ptr(C), ldc, strideC, batch,
                                           _stream(stream), algo)


def conv2d_out_size(H, W, KH, KW, stride=(1, 1), pad=(0, 0), dil=(1, 1)):
    """Output height and width of sgemm_conv2d (floor division)."""
    return ((H + 2 * pad[0] - dil[0] * (KH - 1) - 1) // stride[0] + 1,
            (W + 2 * pad[1] - dil[1] * (KW - 1) - 1) // stride[1] + 1)


SGEMM_CONV_NO_PAD_COPY = 1
SGEMM_FLAG_NO_A_COPY = 1 << 16
SGEMM_FLAG_B_ROWS_LOADED = 1 << 17
SGEMM_FLAG_PAIRS = 1 << 18
SGEMM_FLAG_NO_PAIRS = 1 << 19


def sgemm_conv2d(X, Wt, Y, alpha=1.0, beta=0.0, stride=(1, 1), pad=(0, 0), dil=(1, 1), stream=None,
                 algo=0, shape=None, flags=None) -> int:
    """Y = alpha * conv2d(X, Wt) + beta * Y; X NCHW, Wt OIHW, Y NCHW, fp32 device tensors
    (or addresses, with ``shape`` = (nb, C, H, W, F, KH, KW)).  ``flags`` given: sgemm_conv2d_ex."""
    if shape is None:
        nb, C, H, W = X.shape
        F, _, KH, KW = Wt.shape
    else:
        nb, C, H, W, F, KH, KW = shape
    args = (nb, C, H, W, F, KH, KW, stride[0], stride[1], pad[0], pad[1], dil[0], dil[1],
            alpha, _ptr(X), _ptr(Wt), beta, _ptr(Y), _stream(stream), algo)
    if flags is None:
        return library().sgemm_conv2d(*args)
    return library().sgemm_conv2d_ex(*args, flags)


def sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, algo=0) -> int:
    """Host-buffer entry point; A, B, C are host addresses (ints) or numpy arrays."""
    def hp(x):
        if x is None or isinstance(x, int):
            return x
        if hasattr(x, "ctypes"):
            return x.ctypes.data
        return int(x.data_ptr())
    return library().sgemm_host(M, N, K, alpha, hp(A), lda, hp(B), ldb, beta, hp(C), ldc, algo)


_PLAN_KEYS = ["path", "tile_m", "tile_n", "splits", "units", "grid", "stages", "vec_a", "vec_b",
              "ws_bytes", "tail_tiles", "wide", "pairs"]


def sgemm_host_blocks(M, N, K, lda=None, ldb=None, ldc=None, alpha=1.0, beta=0.0, algo=0, num_sms=0):
    """(axis, sizes): how sgemm_host cuts the call (axis 0: row blocks of C,
    1: column blocks; one size = one GEMM)."""
    lda = max(1, K) if lda is None else lda
    ldb = max(1, N) if ldb is None else ldb
    ldc = max(1, N) if ldc is None else ldc
    axis = ctypes.c_int(0)
    buf = (ctypes.c_int * 16)()
    n = library().sgemm_host_blocks(M, N, K, lda, ldb, ldc, alpha, beta, algo, num_sms, ctypes.byref(axis), buf, 16)
    if n < 0:
        raise SgemmError("sgemm_host_blocks", n)
    return axis.value, list(buf)[:n]


def sgemm_plan_info(M, N, K, A=0, lda=None, B=0, ldb=None, C=0, ldc=None, algo=0, splits=0,
                    flags=0, alpha=1.0, beta=0.0, num_sms=0) -> dict:
    lda = max(1, K) if lda is None else lda
    ldb = max(1, N) if ldb is None else ldb
    ldc = max(1, N) if ldc is None else ldc
    buf = (ctypes.c_int * len(_PLAN_KEYS))()
    rc = library().sgemm_plan_info(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, algo, splits,
                                   flags, alpha, beta, num_sms, buf, len(_PLAN_KEYS))
    if rc != 0:
        raise SgemmError("sgemm_plan_info", rc)
    return dict(zip(_PLAN_KEYS, list(buf)))


def sgemm_check_status(stream=None) -> int:
    return library().sgemm_check_status(_stream(stream))


def sgemm_status_string(status: int) -> str:
    try:
        return library().sgemm_status_string(int(status)).decode()
    except Exception:  # library missing: still describe the code
        return f"status {status}"


def sgemm_tf32_mma_rate(n: int = 256, iters: int = 20000, stream=None) -> float:
    """Raw tf32 TFLOP/s of the tensor cores on the 3xTF32 kernel's MMA form."""
    out = ctypes.c_double(0.0)
    rc = library().sgemm_tf32_mma_rate(n, iters, _stream(stream), ctypes.byref(out))
    if rc != 0:
        raise SgemmError("sgemm_tf32_mma_rate", rc)
    return out.value


def sgemm_ffma_rate(packed: bool = True, iters: int = 20000, stream=None) -> float:
    """fp32 FMA TFLOP/s of the CUDA cores (packed fma.rn.f32x2 or scalar)."""
    out = ctypes.c_double(0.0)
    rc = library().sgemm_ffma_rate(1 if packed else 0, iters, _stream(stream), ctypes.byref(out))
    if rc != 0:
        raise SgemmError("sgemm_ffma_rate", rc)
    return out.value


def sgemm_release() -> int:
    return library().sgemm_release()


def sgemm_version() -> int:
    return library().sgemm_version()


def sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, splits=0) -> int:
    """Allocation-free 3xTF32 entry point (split-K scratch in a fixed library array)."""
    return library().sgemm_noalloc(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                                   _stream(stream), splits)


def sgemm_noalloc_debug_flags(flags: int) -> int:
    """Test hook: debug flags consumed by the next sgemm_noalloc GEMM call."""
    return library().sgemm_noalloc_debug_flags(flags)


# ------------------------------------------------------- torch convenience

def matmul(A, B, C=None, alpha: float = 1.0, beta: float = 0.0, algo: int = SGEMM_ALGO_AUTO,
           splits: int = 0, stream=None):
    """C = alpha*A@B + beta*C for row-major float32 CUDA tensors (unit inner stride).

    Allocates C (uninitialised, beta must then be 0) when it is None.  Runs on
    the current torch stream unless ``stream`` is given; raises SgemmError on a
    non-zero status.  Returns C.
    """
    import torch
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{name} must be a float32 CUDA tensor")
        if t.numel() and t.stride(1) != 1:
            raise ValueError(f"{name} must have unit inner stride (row-major)")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if tuple(C.shape) != (M, N) or C.dtype != torch.float32 or not C.is_cuda:
        raise ValueError("C must be a float32 CUDA tensor of shape (M, N)")
    if C.numel() and C.stride(1) != 1:
        raise ValueError("C must have unit inner stride (row-major)")
    lda = A.stride(0) if M > 1 else max(1, K)
    ldb = B.stride(0) if K > 1 else max(1, N)
    ldc = C.stride(0) if M > 1 else max(1, N)
    st = stream if stream is not None else torch.cuda.current_stream(A.device)
    rc = sgemm_ex(M, N, K, alpha, A, max(lda, max(1, K)), B, max(ldb, max(1, N)), beta, C,
                  max(ldc, max(1, N)), st, algo, splits, 0)
    if rc != 0:
        raise SgemmError("sgemm_ex", rc)
    return C
