"""Seeded synthetic SGEMM workloads: shapes, alpha/beta and input generators.

This module holds no arithmetic of the GEMM itself; it only draws inputs.
Both the CUDA path (tests, bench) and the float64 oracle are fed from here.

Shapes follow the workloads the pages measure:
  * square 256/1024/5120 and a square sweep: "NVIDIA_SGEMM_PRACTICE"
    (overview table, matrix size 5120; run section, size sweep) and
    "matmul_opt.cu" (MATRIX_SIZE 1024);
  * six skinny im2col-shaped products (M, N, K) from the Results table of
    "UNIVERSAL_SGEMM_CUDA" (Quick Run / Results: ./sgemm M N K GEMM_MODE).
The pages publish no input data; the recipes here are:
  * U[-1, 1): numpy PCG64 ``random(dtype=float32) * 2 - 1`` (exact in float32);
  * ReLU(N(0, 1)) for the im2col B operand (activations after a ReLU), drawn
    with ``standard_normal(dtype=float32)`` then max(0, x).
Seeds: 20260000 + 1000 * config index + shape index; A, B, C are drawn in that
order from one generator.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20260000

SKINNY_SHAPES = [
    (32, 1605632, 27),
    (384, 14161, 1152),
    (256, 43264, 1152),
    (64, 1605632, 147),
    (64, 559104, 147),
    (256, 50176, 1024),
]
SWEEP_SIZES = [2048, 4096, 8192, 12288, 16384]


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    seed: int
    b_dist: str = "uniform"      # "uniform" or "relu_normal"
    c_init: str = "uniform"      # "uniform", "nan" (C must not be read), "none"
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def compulsory_bytes(self) -> float:
        """Bytes every implementation must move to/from HBM at least once."""
        c_passes = 2 if self.beta != 0 else 1
        return 4.0 * (self.M * self.K + self.K * self.N + c_passes * self.M * self.N)


def _cfg_seed(cfg: int, shape: int) -> int:
    return SEED_BASE + 1000 * cfg + shape


WORKLOADS: dict[str, Workload] = {}


def _add(w: Workload) -> None:
    WORKLOADS[w.name] = w


_add(Workload("square256", 256, 256, 256, 1.0, 0.0, _cfg_seed(0, 0), c_init="nan",
              note="M=N=K=256, alpha=1, beta=0, C pre-filled with NaN"))
_add(Workload("square1024", 1024, 1024, 1024, 1.5, 0.5, _cfg_seed(1, 0),
              note="M=N=K=1024, alpha=1.5, beta=0.5"))
_add(Workload("ragged1023x1021x1025", 1023, 1021, 1025, 1.5, 0.5, _cfg_seed(1, 1),
              note="M=1023 N=1021 K=1025 packed, alpha=1.5, beta=0.5"))
_add(Workload("square5120", 5120, 5120, 5120, 1.0, 0.5, _cfg_seed(2, 0),
              note="M=N=K=5120, alpha=1, beta=0.5 (size of the pages' headline table)"))
for _i, (_m, _n, _k) in enumerate(SKINNY_SHAPES):
    _add(Workload(f"skinny{_m}x{_n}x{_k}", _m, _n, _k, 1.0, 0.0, _cfg_seed(3, _i),
                  b_dist="relu_normal", c_init="none",
                  note="im2col-shaped, A~U[-1,1), B=ReLU(N(0,1)), alpha=1, beta=0"))
for _i, _s in enumerate(SWEEP_SIZES):
    _add(Workload(f"sweep{_s}", _s, _s, _s, 1.0, 0.0, _cfg_seed(4, _i), c_init="none",
                  note="square sweep, alpha=1, beta=0"))


def uniform(rng: np.random.Generator, n: int) -> np.ndarray:
    """n float32 values, U[-1, 1) on the 2^-23 grid."""
    return rng.random(n, dtype=np.float32) * np.float32(2) - np.float32(1)


def relu_normal(rng: np.random.Generator, n: int) -> np.ndarray:
    x = rng.standard_normal(n, dtype=np.float32)
    return np.maximum(x, np.float32(0))


@dataclass
class Problem:
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    A: np.ndarray            # (M, lda) float32
    B: np.ndarray            # (K, ldb) float32
    C: np.ndarray            # (M, ldc) float32 (initial contents)
    lda: int
    ldb: int
    ldc: int


def make_problem(w: Workload | str, lda: int | None = None, ldb: int | None = None,
                 ldc: int | None = None, pad_value: float = np.nan) -> Problem:
    """Materialise a workload on the host.

    Leading dimensions default to the packed ones. Padding columns (beyond K,
    N) are filled with ``pad_value`` so that a kernel reading them is caught.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    rng = np.random.default_rng(w.seed)
    lda = w.K if lda is None else lda
    ldb = w.N if ldb is None else ldb
    ldc = w.N if ldc is None else ldc
    A = np.full((w.M, max(lda, 1)), pad_value, dtype=np.float32)
    B = np.full((w.K, max(ldb, 1)), pad_value, dtype=np.float32)
    C = np.full((w.M, max(ldc, 1)), pad_value, dtype=np.float32)
    A[:, :w.K] = uniform(rng, w.M * w.K).reshape(w.M, w.K)
    if w.b_dist == "relu_normal":
        B[:, :w.N] = relu_normal(rng, w.K * w.N).reshape(w.K, w.N)
    else:
        B[:, :w.N] = uniform(rng, w.K * w.N).reshape(w.K, w.N)
    if w.c_init == "uniform":
        C[:, :w.N] = uniform(rng, w.M * w.N).reshape(w.M, w.N)
    elif w.c_init == "nan":
        C[:, :w.N] = np.nan
    else:
        C[:, :w.N] = 0.0
    return Problem(w.M, w.N, w.K, w.alpha, w.beta, A, B, C, lda, ldb, ldc)


def random_problem(M: int, N: int, K: int, alpha: float = 1.0, beta: float = 0.0,
                   seed: int = 1, lda: int | None = None, ldb: int | None = None,
                   ldc: int | None = None, pad_value: float = np.nan) -> Problem:
    """Ad-hoc U[-1,1) problem of any shape (used by the shape sweeps of the tests)."""
    w = Workload(f"adhoc{M}x{N}x{K}", M, N, K, alpha, beta, seed)
    return make_problem(w, lda, ldb, ldc, pad_value)


# ------------------------------------------------------------ convolutions
# The layers whose im2col lowering gives the skinny shapes above (M = filters,
# K = channels * KH * KW, N = images * output pixels).  The pages list only the
# lowered shapes; these geometries reproduce them exactly (the 64 x 559104 x 147
# shape has no square-image layer and stays a GEMM workload).  Inputs: X =
# ReLU(N(0, 1)) (the activations the B operand stands for), the filter
# U[-1, 1); seeds 20265000 + layer index; X then the filter from one generator.

@dataclass(frozen=True)
class ConvLayer:
    name: str
    nb: int
    C: int
    H: int
    W: int
    F: int
    KH: int
    KW: int
    stride: int
    pad: int
    seed: int
    gemm: str  # the skinny workload its im2col lowering is

    @property
    def out_hw(self) -> tuple[int, int]:
        return ((self.H + 2 * self.pad - self.KH) // self.stride + 1,
                (self.W + 2 * self.pad - self.KW) // self.stride + 1)

    @property
    def gemm_mnk(self) -> tuple[int, int, int]:
        oh, ow = self.out_hw
        return self.F, self.nb * oh * ow, self.C * self.KH * self.KW

    @property
    def flops(self) -> float:
        m, n, k = self.gemm_mnk
        return 2.0 * m * n * k

    @property
    def compulsory_bytes(self) -> float:
        """Input, filter and output once (beta = 0: the output is only written)."""
        oh, ow = self.out_hw
        return 4.0 * (self.nb * self.C * self.H * self.W + self.F * self.C * self.KH * self.KW +
                      self.nb * self.F * oh * ow)

    def note(self) -> str:
        m, n, k = self.gemm_mnk
        return (f"conv2d NCHW {self.nb}x{self.C}x{self.H}x{self.W}, {self.F} filters {self.KH}x{self.KW}, "
                f"stride {self.stride}, pad {self.pad}, alpha=1, beta=0; im2col GEMM {m}x{n}x{k} ({self.gemm})")


CONV_LAYERS: dict[str, ConvLayer] = {}
for _i, (_nb, _c, _h, _w, _f, _k, _s, _p, _g) in enumerate([
        (32, 3, 224, 224, 32, 3, 1, 1, "skinny32x1605632x27"),
        (1, 128, 121, 121, 384, 3, 1, 0, "skinny384x14161x1152"),
        (1, 128, 210, 210, 256, 3, 1, 0, "skinny256x43264x1152"),
        (32, 3, 224, 224, 64, 7, 1, 3, "skinny64x1605632x147"),
        (1, 64, 227, 227, 256, 4, 1, 0, "skinny256x50176x1024")]):
    _name = f"conv{_nb}x{_c}x{_h}x{_w}f{_f}k{_k}p{_p}"
    CONV_LAYERS[_name] = ConvLayer(_name, _nb, _c, _h, _w, _f, _k, _k, _s, _p, SEED_BASE + 5000 + _i, _g)


def make_conv_inputs(layer: ConvLayer | str) -> tuple[np.ndarray, np.ndarray]:
    """(X, filter) of a convolution layer, float32 NCHW and OIHW."""
    if isinstance(layer, str):
        layer = CONV_LAYERS[layer]
    rng = np.random.default_rng(layer.seed)
    X = relu_normal(rng, layer.nb * layer.C * layer.H * layer.W).reshape(layer.nb, layer.C, layer.H, layer.W)
    Wt = uniform(rng, layer.F * layer.C * layer.KH * layer.KW).reshape(layer.F, layer.C, layer.KH, layer.KW)
    return X, Wt
