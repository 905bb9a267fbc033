"""Pins for the float64 convolution oracle (``oracle.conv2d_ref``).

The pages list the im2col GEMM shapes of convolution layers but do not
define the layer; the oracle states the usual definition (cross-correlation,
NCHW input, OIHW filter, zero padding, stride and dilation).  Each pin holds
it against something outside the oracle's code:

- a 1x1 filter is a plain matrix product (numpy float64 ``@``);
- a one-hot filter copies a shifted, strided, dilated window of the input,
  formed here by numpy slicing of a zero-padded array;
- a single-channel layer is ``scipy.signal.correlate2d`` (a library routine,
  which does not flip the filter);
- stride s is the stride-1 result sampled every s pixels, and dilation d is a
  filter with d - 1 zeros inserted between its taps (invariants of the
  definition);
- an all-ones input gives each output the sum of the filter taps that fall
  inside the image (closed form, counted per tap).

The last test builds wrong variants of the oracle (filter flipped, padding on
one side only, dilation ignored) and shows that each fails at least one pin.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_05_gb300.workloads import uniform


def _rand(shape, seed):
    return uniform(np.random.default_rng(seed), int(np.prod(shape))).reshape(shape)


def _close(got, want, scale, rel=1e-12):
    return bool(np.all(np.abs(got - want) <= rel * scale + 1e-300))


# ---------------------------------------------------------------- pin bodies

def pin_1x1_is_matmul(plant=0) -> bool:
    """A 1x1 filter with stride 1 and no padding is Wt (F x C) times each
    image as a C x (H W) matrix; the scale is |Wt| times |X|."""
    nb, C, H, W, F = 2, 5, 6, 7, 4
    X, Wt = _rand((nb, C, H, W), 1), _rand((F, C, 1, 1), 2)
    ref, scale = oracle.conv2d_ref(1.5, X, Wt, plant=plant)
    w = Wt.reshape(F, C).astype(np.float64)
    ok = True
    for b in range(nb):
        x = X[b].reshape(C, H * W).astype(np.float64)
        want = (1.5 * (w @ x)).reshape(F, H, W)
        want_s = (1.5 * (np.abs(w) @ np.abs(x))).reshape(F, H, W)
        ok &= _close(ref[b], want, want_s) and _close(scale[b], want_s, want_s)
    return ok


def pin_one_hot_filter(plant=0) -> bool:
    """A filter with one tap of 1 at (f mod C, kh0, kw0) off the centre
    copies the input window that tap sees, exactly, zeros outside the image."""
    nb, C, H, W, F, KH, KW = 2, 3, 11, 9, 5, 3, 4
    stride, pad, dil = (2, 1), (2, 1), (2, 3)
    X = _rand((nb, C, H, W), 3)
    OH, OW = oracle.conv2d_out_size(H, W, KH, KW, stride, pad, dil)
    ok = True
    for kh0, kw0 in ((0, 1), (2, 3), (1, 0)):
        Wt = np.zeros((F, C, KH, KW), np.float32)
        for f in range(F):
            Wt[f, f % C, kh0, kw0] = 1.0
        ref, _ = oracle.conv2d_ref(1.0, X, Wt, stride=stride, pad=pad, dil=dil, plant=plant)
        Xp = np.zeros((nb, C, H + 2 * pad[0] + 64, W + 2 * pad[1] + 64), np.float64)
        Xp[:, :, pad[0]:pad[0] + H, pad[1]:pad[1] + W] = X
        r0, c0 = kh0 * dil[0], kw0 * dil[1]
        win = Xp[:, :, r0:r0 + stride[0] * OH:stride[0], c0:c0 + stride[1] * OW:stride[1]]
        want = np.stack([win[:, f % C] for f in range(F)], axis=1)
        ok &= bool(np.array_equal(ref, want))
    return ok


def pin_scipy_correlate2d(plant=0) -> bool:
    """One channel, one filter, stride 1: scipy's 2-D cross-correlation of
    the zero-padded image ('valid' mode)."""
    signal = pytest.importorskip("scipy.signal")
    H, W, KH, KW = 13, 10, 5, 3
    ok = True
    for pad in ((0, 0), (2, 1)):
        X, Wt = _rand((1, 1, H, W), 4), _rand((1, 1, KH, KW), 5)
        ref, scale = oracle.conv2d_ref(1.0, X, Wt, pad=pad, plant=plant)
        xp = np.pad(X[0, 0].astype(np.float64), ((pad[0], pad[0]), (pad[1], pad[1])))
        want = signal.correlate2d(xp, Wt[0, 0].astype(np.float64), mode="valid")
        want_s = signal.correlate2d(np.abs(xp), np.abs(Wt[0, 0]).astype(np.float64), mode="valid")
        ok &= want.shape == ref.shape[2:] and _close(ref[0, 0], want, want_s)
    return ok


def pin_stride_is_subsampling(plant=0) -> bool:
    """Stride (sh, sw) gives the stride-1 output at every sh-th row and
    sw-th column, bit for bit."""
    X, Wt = _rand((2, 3, 12, 13), 6), _rand((4, 3, 3, 2), 7)
    full, _ = oracle.conv2d_ref(0.75, X, Wt, pad=(1, 1), plant=plant)
    ok = True
    for st in ((2, 3), (3, 1)):
        ref, _ = oracle.conv2d_ref(0.75, X, Wt, stride=st, pad=(1, 1), plant=plant)
        ok &= bool(np.array_equal(ref, full[:, :, ::st[0], ::st[1]]))
    return ok


def pin_dilation_is_zero_inserted_filter(plant=0) -> bool:
    """Dilation (dh, dw) equals dilation 1 with dh - 1 and dw - 1 zero rows
    and columns between the filter taps."""
    X, Wt = _rand((1, 2, 14, 15), 8), _rand((3, 2, 3, 3), 9)
    dh, dw = 2, 3
    Wz = np.zeros((3, 2, 1 + (3 - 1) * dh, 1 + (3 - 1) * dw), np.float32)
    Wz[:, :, ::dh, ::dw] = Wt
    ref, scale = oracle.conv2d_ref(1.0, X, Wt, pad=(1, 2), dil=(dh, dw), plant=plant)
    want, _ = oracle.conv2d_ref(1.0, X, Wz, pad=(1, 2), plant=0)
    return ref.shape == want.shape and _close(ref, want, scale)


def pin_ones_input_counts_taps(plant=0) -> bool:
    """X = 1 everywhere: each output is the sum of the taps whose input
    position lies inside the image, counted tap by tap here."""
    nb, C, H, W, F, KH, KW = 1, 2, 6, 5, 3, 3, 4
    stride, pad, dil = (1, 2), (2, 1), (1, 1)
    X = np.ones((nb, C, H, W), np.float32)
    Wt = _rand((F, C, KH, KW), 10)
    ref, scale = oracle.conv2d_ref(1.0, X, Wt, stride=stride, pad=pad, dil=dil, plant=plant)
    OH, OW = ref.shape[2:]
    want = np.zeros((F, OH, OW))
    for oh in range(OH):
        rows = [kh for kh in range(KH) if 0 <= oh * stride[0] - pad[0] + kh * dil[0] < H]
        for ow in range(OW):
            cols = [kw for kw in range(KW) if 0 <= ow * stride[1] - pad[1] + kw * dil[1] < W]
            want[:, oh, ow] = Wt[:, :, rows][:, :, :, cols].astype(np.float64).sum(axis=(1, 2, 3))
    return _close(ref[0], want, scale[0])


PINS = [pin_1x1_is_matmul, pin_one_hot_filter, pin_scipy_correlate2d, pin_stride_is_subsampling,
        pin_dilation_is_zero_inserted_filter, pin_ones_input_counts_taps]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_conv_pin_holds(oracle_mod, pin):
    assert pin(0), pin.__doc__


def test_conv_beta_and_alpha(oracle_mod):
    """beta == 0 does not read Y (NaN there stays out); the beta term and
    alpha scale as in the GEMM oracle."""
    X, Wt = _rand((2, 3, 8, 8), 11), _rand((4, 3, 3, 3), 12)
    Y = _rand((2, 4, 6, 6), 13)
    base, bscale = oracle.conv2d_ref(1.0, X, Wt)
    nan_y = np.full_like(Y, np.nan)
    r0, _ = oracle.conv2d_ref(2.0, X, Wt, beta=0.0, Y=nan_y)
    assert np.all(np.isfinite(r0)) and np.array_equal(r0, 2.0 * base)
    r1, s1 = oracle.conv2d_ref(2.0, X, Wt, beta=-0.5, Y=Y)
    assert np.array_equal(r1, 2.0 * base + (-0.5) * Y.astype(np.float64))
    assert np.array_equal(s1, 2.0 * bscale + np.abs(0.5 * Y.astype(np.float64)))


def test_conv_rejects_bad_arguments(oracle_mod):
    X, Wt = _rand((1, 2, 4, 4), 14), _rand((1, 3, 3, 3), 15)
    with pytest.raises(ValueError):
        oracle.conv2d_ref(1.0, X, Wt)  # channel mismatch
    with pytest.raises(ValueError):
        oracle.conv2d_ref(1.0, X, _rand((1, 2, 5, 5), 16))  # filter larger than the image


@pytest.mark.parametrize("plant,what", [(5, "filter flipped"), (6, "padding on one side only"),
                                        (7, "dilation ignored")])
def test_each_planted_conv_mistake_fails_a_pin(oracle_mod, plant, what):
    oracle.build(plant)
    failed = [p.__name__ for p in PINS if not p(plant)]
    assert failed, f"no pin catches the planted mistake: {what}"
