"""The seeded synthetic inputs that the tests and the benchmark share.

The input recipe is part of every measurement: shapes, alpha and beta of
each workload, seeds, the U[-1, 1) grid of the uniform operands and the
ReLU(N(0, 1)) activations that stand in for an im2col B.  These checks keep
it what the design states, and keep every convolution layer an exact
lowering of the GEMM workload it stands for.
"""
import numpy as np
import pytest

from dense_fp32_matrix_05_gb300 import workloads as wl


def test_workload_table():
    W = wl.WORKLOADS
    assert (W["square256"].M, W["square256"].alpha, W["square256"].beta, W["square256"].c_init) == \
        (256, 1.0, 0.0, "nan")
    assert (W["square1024"].alpha, W["square1024"].beta) == (1.5, 0.5)
    r = W["ragged1023x1021x1025"]
    assert (r.M, r.N, r.K, r.alpha, r.beta) == (1023, 1021, 1025, 1.5, 0.5)
    h = W["square5120"]
    assert (h.M, h.N, h.K, h.alpha, h.beta) == (5120, 5120, 5120, 1.0, 0.5)
    skinny = [n for n in W if n.startswith("skinny")]
    assert [(W[n].M, W[n].N, W[n].K) for n in skinny] == wl.SKINNY_SHAPES
    assert all(W[n].b_dist == "relu_normal" and W[n].beta == 0.0 and W[n].alpha == 1.0 for n in skinny)
    assert [W[f"sweep{s}"].M for s in wl.SWEEP_SIZES] == [2048, 4096, 8192, 12288, 16384]
    # seeds: 20260000 + 1000 * configuration + shape index, all distinct
    assert W["square256"].seed == 20260000 and W["ragged1023x1021x1025"].seed == 20261001
    assert W["skinny64x559104x147"].seed == 20263004 and W["sweep16384"].seed == 20264004
    assert len({w.seed for w in W.values()}) == len(W)


def test_compulsory_bytes():
    w = wl.WORKLOADS["square5120"]           # beta != 0: C is read and written
    assert w.compulsory_bytes == 4.0 * 3 * 5120 * 5120 + 4.0 * 5120 * 5120
    s = wl.WORKLOADS["skinny32x1605632x27"]  # beta = 0: C is only written
    assert s.compulsory_bytes == 4.0 * (32 * 27 + 27 * 1605632 + 32 * 1605632)


def test_uniform_grid_and_range():
    x = wl.uniform(np.random.default_rng(1), 1 << 16)
    assert x.dtype == np.float32
    assert x.min() >= -1.0 and x.max() < 1.0
    scaled = x.astype(np.float64) * 2.0 ** 23
    assert np.array_equal(scaled, np.round(scaled))                  # on the 2^-23 grid
    assert abs(float(x.mean())) < 0.02 and abs(float((x < 0).mean()) - 0.5) < 0.02


def test_relu_normal_activations():
    x = wl.relu_normal(np.random.default_rng(2), 1 << 16)
    assert x.dtype == np.float32 and x.min() == 0.0
    zero = float((x == 0).mean())
    assert abs(zero - 0.5) < 0.02                                    # half the draws clip to 0
    assert abs(float(x[x > 0].mean()) - np.sqrt(2 / np.pi)) < 0.02   # half-normal mean


def test_make_problem_is_deterministic_and_padded():
    p1 = wl.make_problem("square256", lda=260, ldb=257, ldc=300, pad_value=-7.0)
    p2 = wl.make_problem("square256", lda=260, ldb=257, ldc=300, pad_value=-7.0)
    for a, b in ((p1.A, p2.A), (p1.B, p2.B)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.all(p1.A[:, 256:] == -7.0) and np.all(p1.B[:, 256:] == -7.0) and np.all(p1.C[:, 256:] == -7.0)
    assert np.all(np.isnan(p1.C[:, :256]))                           # C must not be read at beta = 0
    q = wl.make_problem("square1024")
    assert np.all(np.isfinite(q.C)) and q.C.min() >= -1.0            # beta != 0: uniform C
    # the packed matrices are the first rows of the same draws whatever the ld
    packed = wl.make_problem("square256")
    assert np.array_equal(packed.A, p1.A[:, :256]) and np.array_equal(packed.B, p1.B[:, :256])


@pytest.mark.parametrize("name", list(wl.CONV_LAYERS))
def test_conv_layers_lower_to_their_gemm_workloads(name):
    layer = wl.CONV_LAYERS[name]
    g = wl.WORKLOADS[layer.gemm]
    assert layer.gemm_mnk == (g.M, g.N, g.K)
    assert layer.flops == g.flops
    X, Wt = wl.make_conv_inputs(name) if layer.nb * layer.C * layer.H * layer.W < 2e6 else (None, None)
    if X is not None:
        assert X.shape == (layer.nb, layer.C, layer.H, layer.W) and X.min() >= 0.0
        assert Wt.shape == (layer.F, layer.C, layer.KH, layer.KW) and Wt.min() >= -1.0 and Wt.max() < 1.0
