"""Float64 CPU oracle for C = alpha*A*B + beta*C on row-major float32 matrices.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The CUDA library and its
Python binding never import it, and it shares no code with them.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, OpenMP over rows). It is
the CPU triple loop matrixMulCPU of "matmul_opt.cu" (cnblogs matmul-opt demo)
extended to the problem statement mysgemm(M,N,K,alpha,A,B,beta,C) of
"NVIDIA_SGEMM_PRACTICE" (section "kernel 1"): leading dimensions, float64
accumulation, the alpha/beta epilogue, and a second sum of |a*b| that gives
each element its error scale.

``within_bound`` is the acceptance rule every GPU result is held to:
|gpu - ref| <= 1e-4 * (|alpha| * sum_k |a_mk * b_kn| + |beta * c_mn|),
compared in float64 against the unrounded float64 reference.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}

#: relative tolerance of the acceptance rule
REL_TOL = 1e-4


def lib_path(plant: int = 0) -> str:
    tag = platform.machine()
    suffix = "" if plant == 0 else f"_plant{plant}"
    return os.path.join(_BUILD, f"liboracle_{tag}{suffix}.so")


def build(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle with the host C compiler; returns the .so path.

    ``plant`` > 0 builds a deliberately wrong variant (used only by the tests
    that show each pin catches a mistake).
    """
    out = lib_path(plant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", f"-DORACLE_PLANT={int(plant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(plant: int = 0) -> ctypes.CDLL:
    with _lock:
        if plant not in _libs:
            lib = ctypes.CDLL(build(plant))
            f = lib.oracle_sgemm_rows
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                          ctypes.c_void_p, ctypes.c_longlong,
                          ctypes.c_void_p, ctypes.c_longlong,
                          ctypes.c_double, ctypes.c_void_p, ctypes.c_longlong,
                          ctypes.c_void_p, ctypes.c_int,
                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            g = lib.oracle_conv2d_nchw
            g.restype = ctypes.c_int
            g.argtypes = ([ctypes.c_int] * 13 + [ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_double, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int])
            lib.oracle_max_threads.restype = ctypes.c_int
            _libs[plant] = lib
        return _libs[plant]


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def sgemm_ref(M: int, N: int, K: int, alpha: float, A, lda: int, B, ldb: int,
              beta: float, C, ldc: int, rows=None, threads: int = 0,
              plant: int = 0):
    """Reference result and error scale for the selected output rows.

    A, B, C are float32 numpy buffers (any shape, C-contiguous) holding the
    row-major matrices with the given leading dimensions; C may be None when
    beta == 0, A and B may be None when alpha == 0 or K == 0.
    ``rows`` (sequence of row indices) restricts the computation to those
    output rows; default: all rows.

    Returns (ref, scale): float64 arrays of shape (len(rows), N).
    ``scale`` = |alpha| * sum_k |A[m,k] * B[k,n]| + |beta * C[m,n]|.
    """
    def as_f32(x):
        if x is None:
            return None
        x = np.ascontiguousarray(x)
        if x.dtype != np.float32:
            raise TypeError("oracle inputs must be float32")
        return x

    A, B, C = as_f32(A), as_f32(B), as_f32(C)
    if rows is None:
        rows_arr = None
        nrows = M
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        nrows = int(rows_arr.size)
    ref = np.empty((nrows, N), dtype=np.float64)
    scale = np.empty((nrows, N), dtype=np.float64)
    rc = _lib(plant).oracle_sgemm_rows(
        int(M), int(N), int(K), float(alpha), _ptr(A), int(lda), _ptr(B), int(ldb),
        float(beta), _ptr(C), int(ldc), _ptr(rows_arr), int(nrows),
        ref.ctypes.data, scale.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_sgemm_rows rejected argument {-rc}")
    return ref, scale


def conv2d_out_size(H: int, W: int, KH: int, KW: int, stride=(1, 1), pad=(0, 0), dil=(1, 1)):
    """Output height and width of a 2-D convolution (floor division)."""
    oh = (H + 2 * pad[0] - dil[0] * (KH - 1) - 1) // stride[0] + 1
    ow = (W + 2 * pad[1] - dil[1] * (KW - 1) - 1) // stride[1] + 1
    return oh, ow


def conv2d_ref(alpha: float, X, Wt, beta: float = 0.0, Y=None, stride=(1, 1), pad=(0, 0),
               dil=(1, 1), threads: int = 0, plant: int = 0):
    """Direct 2-D convolution (no filter flip) of NCHW ``X`` with OIHW
    ``Wt``: Y = alpha * conv(X, Wt) + beta * Y, zero padding.

    The pages give only the GEMM shapes that this layer lowers to through
    im2col (filters x (channels * KH * KW) times (channels * KH * KW) x
    pixels); ``oracle_conv2d_nchw`` in the C file states the definition.
    Returns (ref, scale), float64 arrays nb x F x OH x OW, with the same
    per-element error scale as ``sgemm_ref``.
    """
    X = np.ascontiguousarray(X)
    Wt = np.ascontiguousarray(Wt)
    if X.dtype != np.float32 or Wt.dtype != np.float32:
        raise TypeError("oracle inputs must be float32")
    nb, C, H, W = X.shape
    F, C2, KH, KW = Wt.shape
    if C2 != C:
        raise ValueError("filter channels differ from input channels")
    OH, OW = conv2d_out_size(H, W, KH, KW, stride, pad, dil)
    if OH < 1 or OW < 1:
        raise ValueError("empty output")
    if beta != 0.0:
        Y = np.ascontiguousarray(Y)
        if Y.dtype != np.float32 or Y.shape != (nb, F, OH, OW):
            raise TypeError("Y must be float32 nb x F x OH x OW")
    else:
        Y = None
    ref = np.empty((nb, F, OH, OW), dtype=np.float64)
    scale = np.empty_like(ref)
    rc = _lib(plant).oracle_conv2d_nchw(
        nb, C, H, W, F, KH, KW, int(stride[0]), int(stride[1]), int(pad[0]), int(pad[1]),
        int(dil[0]), int(dil[1]), float(alpha), X.ctypes.data, Wt.ctypes.data, float(beta),
        _ptr(Y), ref.ctypes.data, scale.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_conv2d_nchw rejected argument {-rc}")
    return ref, scale


def within_bound(got, ref, scale, rel: float = REL_TOL):
    """Element-wise acceptance mask of the parity rule.

    |got - ref| <= rel * scale, in float64. An infinite reference must be
    matched exactly; a NaN reference must be matched by NaN.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.asarray(scale, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        ok = np.abs(got - ref) <= rel * scale
    both_nan = np.isnan(got) & np.isnan(ref)
    inf_ref = np.isinf(ref)
    ok = np.where(inf_ref, got == ref, ok)
    return ok | both_nan


def first_failures(got, ref, scale, rel: float = REL_TOL, limit: int = 5):
    """Human-readable description of the first failing elements (or '')."""
    ok = within_bound(got, ref, scale, rel)
    bad = np.argwhere(~ok)
    if bad.size == 0:
        return ""
    lines = [f"{bad.shape[0]} of {ok.size} elements outside the bound"]
    for idx in bad[:limit]:
        t = tuple(int(i) for i in idx)
        lines.append(f"  at {t}: got={np.asarray(got)[t]!r} ref={ref[t]!r} "
                     f"bound={rel * scale[t]!r}")
    return "\n".join(lines)
