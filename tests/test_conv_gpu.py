"""Parity of the implicit-GEMM convolution (sgemm_conv2d) against the
float64 direct-convolution oracle, element by element, through the C ABI.

Each case fills guard bands around Y with a sentinel and checks them after
the call; the acceptance rule is the GEMM one with the sum over the taps
that fall inside the image.
"""
from __future__ import annotations

import numpy as np
import pytest

import dense_fp32_matrix_05_gb300 as pkg
import oracle
from dense_fp32_matrix_05_gb300.workloads import relu_normal, uniform

pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = np.float32(-3.0e33)


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    pkg.library()


def _inputs(nb, C, H, W, F, KH, KW, seed, relu=False):
    rng = np.random.default_rng(seed)
    n = nb * C * H * W
    X = (relu_normal(rng, n) if relu else uniform(rng, n)).reshape(nb, C, H, W)
    Wt = uniform(rng, F * C * KH * KW).reshape(F, C, KH, KW)
    return X, Wt


def _run(X, Wt, Y0, alpha, beta, stride, pad, dil, images=None, algo=0, flags=None):
    """sgemm_conv2d on the device; returns the selected images of Y."""
    import torch
    nb, F, OH, OW = Y0.shape
    dX = torch.from_numpy(np.ascontiguousarray(X)).cuda()
    dW = torch.from_numpy(np.ascontiguousarray(Wt)).cuda()
    buf = torch.full((GUARD + Y0.size + GUARD,), float(SENTINEL), device="cuda")
    buf[GUARD:GUARD + Y0.size] = torch.from_numpy(Y0.reshape(-1)).cuda()
    st = torch.cuda.current_stream()
    rc = pkg.sgemm_conv2d(dX, dW, buf.data_ptr() + GUARD * 4, alpha=alpha, beta=beta, stride=stride, pad=pad,
                          dil=dil, stream=st, shape=X.shape + Wt.shape[:1] + Wt.shape[2:], algo=algo,
                          flags=flags)
    assert rc == 0, rc
    assert pkg.sgemm_check_status(st) == 0
    out = buf.cpu().numpy()
    assert np.all(out[:GUARD] == SENTINEL) and np.all(out[GUARD + Y0.size:] == SENTINEL), "write outside Y"
    Y = out[GUARD:GUARD + Y0.size].reshape(Y0.shape)
    return Y if images is None else Y[images]


def _check(X, Wt, alpha, beta, stride, pad, dil, seed, images=None, algo=0, flags=None):
    nb, C, H, W = X.shape
    F = Wt.shape[0]
    OH, OW = oracle.conv2d_out_size(H, W, Wt.shape[2], Wt.shape[3], stride, pad, dil)
    Y0 = uniform(np.random.default_rng(seed + 1), nb * F * OH * OW).reshape(nb, F, OH, OW)
    got = _run(X, Wt, Y0, alpha, beta, stride, pad, dil, images, algo, flags)
    sel = slice(None) if images is None else images
    ref, scale = oracle.conv2d_ref(alpha, X[sel], Wt, beta, Y0[sel] if beta != 0 else None, stride, pad, dil)
    msg = oracle.first_failures(got, ref, scale)
    assert not msg, msg


# nb, C, H, W, F, KH, KW, stride, pad, dil, alpha, beta
CASES = [
    (2, 3, 17, 19, 32, 3, 3, (1, 1), (1, 1), (1, 1), 1.0, 0.0),      # K = 27: filter rows staged to 16 bytes
    (1, 16, 12, 13, 40, 3, 3, (2, 2), (1, 1), (1, 1), 1.5, 0.5),     # K = 144, ragged filters and pixels
    (3, 3, 23, 23, 64, 7, 7, (2, 2), (3, 3), (1, 1), 1.0, 0.0),      # 7 x 7 stride 2 (K = 147)
    (2, 8, 20, 21, 24, 3, 2, (1, 2), (2, 0), (2, 3), -0.5, 1.0),     # dilation, asymmetric everything
    (4, 32, 9, 9, 130, 1, 1, (1, 1), (0, 0), (1, 1), 1.0, 0.0),      # 1 x 1: a batched GEMM, 130 filters
    (1, 128, 16, 16, 256, 3, 3, (1, 1), (0, 0), (1, 1), 1.0, 0.25),  # K = 1152, few tiles: K slices
    (1, 64, 31, 31, 200, 4, 4, (1, 1), (0, 0), (1, 1), 1.0, 0.0),    # K = 1024
    (5, 4, 6, 5, 3, 5, 5, (1, 1), (2, 2), (1, 1), 2.0, 0.0),         # image smaller than one tile, 3 filters
    (40, 3, 14, 14, 16, 3, 3, (1, 1), (1, 1), (1, 1), 1.0, 0.5),     # many small images: one launch
    (3, 7, 9, 10, 32, 3, 3, (2, 1), (0, 2), (1, 2), 1.0, 0.0),       # K = 63, 32 filters: FFMA form fits
    (2, 2, 37, 41, 5, 5, 3, (1, 3), (2, 1), (2, 1), -1.0, 0.75),     # K = 30, 5 filters, pixels not even
]
# small enough for the FFMA form (F <= 32, K <= 64): run on both paths
FFMA_FITS = [c for c in CASES if c[4] <= 32 and c[1] * c[5] * c[6] <= 64]
ALGOS = [("auto", pkg.SGEMM_ALGO_AUTO), ("tf32x3", pkg.SGEMM_ALGO_TF32X3), ("ffma", pkg.SGEMM_ALGO_FFMA)]


def _case_id(c):
    return (f"b{c[0]}c{c[1]}h{c[2]}w{c[3]}f{c[4]}k{c[5]}x{c[6]}s{c[7][0]}{c[7][1]}"
            f"p{c[8][0]}{c[8][1]}d{c[9][0]}{c[9][1]}")


# every case on AUTO and 3xTF32; on FFMA only where its form applies (the
# library rejects the rest with -20, which test_abi_cpu checks)
PARITY = [pytest.param(c, a, id=f"{n}-{_case_id(c)}") for n, a in ALGOS for c in CASES
          if a != pkg.SGEMM_ALGO_FFMA or c in FFMA_FITS]


@pytest.mark.parametrize("case,algo", PARITY)
def test_conv2d_parity(case, algo):
    nb, C, H, W, F, KH, KW, stride, pad, dil, alpha, beta = case
    X, Wt = _inputs(nb, C, H, W, F, KH, KW, seed=sum(case[:7]))
    _check(X, Wt, alpha, beta, stride, pad, dil, seed=nb * 1000 + F, algo=algo)


PADDED_TAPS = [c for c in CASES if c[1] % 16 != 0 and (c[8][0] or c[8][1])]


GATHER = [pytest.param(c, a, id=f"{n}-b{c[0]}c{c[1]}f{c[4]}k{c[5]}x{c[6]}p{c[8][0]}{c[8][1]}")
          for n, a in (("tf32x3", pkg.SGEMM_ALGO_TF32X3), ("ffma", pkg.SGEMM_ALGO_FFMA)) for c in PADDED_TAPS
          if a != pkg.SGEMM_ALGO_FFMA or c in FFMA_FITS]


@pytest.mark.parametrize("case,algo", GATHER)
def test_conv2d_bounds_checked_gather(case, algo):
    """Padded layers without the zero-bordered input copy: the gather checks
    every tap against the image (the path a copy over 1 GiB also takes)."""
    nb, C, H, W, F, KH, KW, stride, pad, dil, alpha, beta = case
    X, Wt = _inputs(nb, C, H, W, F, KH, KW, seed=sum(case[:7]) + 5)
    _check(X, Wt, alpha, beta, stride, pad, dil, seed=nb * 1000 + F + 5, algo=algo,
           flags=pkg.SGEMM_CONV_NO_PAD_COPY)


@pytest.mark.parametrize("layer", [(32, 3, 224, 224, 32, 3, 3, 1, 1), (32, 3, 224, 224, 64, 7, 7, 1, 3),
                                   (1, 128, 121, 121, 384, 3, 3, 1, 0)],
                         ids=["32x3x224x224-f32k3", "32x3x224x224-f64k7", "1x128x121x121-f384k3"])
@pytest.mark.parametrize("algo", [pkg.SGEMM_ALGO_AUTO, pkg.SGEMM_ALGO_TF32X3], ids=["auto", "tf32x3"])
def test_conv2d_full_size_layers(layer, algo):
    """The layers whose im2col GEMMs are the skinny benchmark shapes
    (32 x 1605632 x 27, 64 x 1605632 x 147, 384 x 14161 x 1152), with ReLU'd
    normal inputs; the oracle checks the first and last image."""
    nb, C, H, W, F, KH, KW, s, p = layer
    X, Wt = _inputs(nb, C, H, W, F, KH, KW, seed=F + KH, relu=True)
    images = [0, nb - 1] if nb > 1 else [0]
    _check(X, Wt, 1.0, 0.0, (s, s), (p, p), (1, 1), seed=7, images=images, algo=algo)


@pytest.mark.parametrize("C,algo", [(4, pkg.SGEMM_ALGO_TF32X3), (16, pkg.SGEMM_ALGO_TF32X3),
                                    (4, pkg.SGEMM_ALGO_FFMA)], ids=["taps-tf32x3", "channels-tf32x3", "ffma"])
def test_conv2d_special_values(C, algo):
    """An infinite input pixel gives +-Inf (or NaN where the taps' signs
    clash) in the outputs that see it, as fp64 arithmetic does; the tensor
    path's NaN recompute on the CUDA cores walks the taps of the window in
    its k order."""
    X, Wt = _inputs(2, C, 10, 11, 20, 3, 3, seed=91)
    X[0, 1, 4, 5] = np.inf
    X[1, 2, 0, 0] = -np.inf
    _check(X, Wt, 1.0, 0.0, (1, 1), (1, 1), (1, 1), seed=92, algo=algo)


def test_conv2d_alpha_zero_and_no_channels():
    """alpha == 0 leaves beta * Y without reading X or the filter."""
    import torch
    nb, F, OH, OW = 2, 5, 6, 7
    Y0 = uniform(np.random.default_rng(93), nb * F * OH * OW).reshape(nb, F, OH, OW)
    dY = torch.from_numpy(Y0.copy()).cuda()
    rc = pkg.sgemm_conv2d(None, None, dY, alpha=0.0, beta=0.5, shape=(nb, 3, OH + 2, OW + 2, F, 3, 3))
    assert rc == 0
    torch.cuda.synchronize()
    assert np.array_equal(dY.cpu().numpy(), (np.float32(0.5) * Y0).astype(np.float32))
    rc = pkg.sgemm_conv2d(None, None, dY, alpha=1.0, beta=0.0, shape=(nb, 0, OH + 2, OW + 2, F, 3, 3))
    assert rc == 0
    torch.cuda.synchronize()
    assert np.all(dY.cpu().numpy() == 0)


def test_conv2d_matches_strided_batched_gemm_on_1x1():
    """A 1 x 1 convolution and the strided batch of the same GEMMs (filter
    shared, one C x HW image per matrix) run the same kernel schedule and
    give the same bits."""
    import torch
    nb, C, H, W, F = 3, 64, 20, 20, 96
    X, Wt = _inputs(nb, C, H, W, F, 1, 1, seed=94)
    dX = torch.from_numpy(X).cuda()
    dW = torch.from_numpy(Wt).cuda()
    Y1 = torch.zeros((nb, F, H, W), device="cuda")
    Y2 = torch.zeros((nb, F, H, W), device="cuda")
    assert pkg.sgemm_conv2d(dX, dW, Y1) == 0
    HW = H * W
    assert pkg.sgemm_strided_batched(0, 0, F, HW, C, 1.0, dW, C, 0, dX, HW, C * HW, 0.0, Y2, HW, F * HW, nb) == 0
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
