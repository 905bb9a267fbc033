"""Pins for the float64 oracle, each independent of the oracle's own code.

Every pin compares the oracle with something fixed by the pages or by the
mathematics: closed forms (identity, permutation, constant matrices), exact
integer arithmetic (numpy int64), exact rational arithmetic (fractions), an
independent float64 formulation (numpy/BLAS matmul), and the BLAS reading of
beta == 0 / alpha == 0.  The last test builds deliberately wrong variants of
the oracle (transposed A, dropped beta term, dropped last k, swapped
alpha/beta) and shows that each one fails at least one pin.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_fp32_matrix_05_gb300.workloads import random_problem, uniform

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ref(p, plant=0, rows=None):
    return oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb,
                            p.beta, p.C, p.ldc, rows=rows, plant=plant)


# ---------------------------------------------------------------- pin bodies
# Each pin takes a ``plant`` argument so the planted-mistake test can rerun it
# against a wrong build of the oracle. A pin returns True when it holds.

def pin_identity(plant=0) -> bool:
    """A = I (K = M): C = alpha*B + beta*C exactly for power-of-two alpha, beta."""
    M = N = K = 37
    rng = np.random.default_rng(11)
    A = np.eye(M, K, dtype=np.float32)
    B = uniform(rng, K * N).reshape(K, N)
    C = uniform(rng, M * N).reshape(M, N)
    ref, _ = oracle.sgemm_ref(M, N, K, 2.0, A, K, B, N, 0.5, C, N, plant=plant)
    # exact: 2*b and 0.5*c are exact; the sum of two values on the 2^-25 grid
    # below 4 in magnitude is exact in float64
    want = 2.0 * B.astype(np.float64) + 0.5 * C.astype(np.float64)
    ok_left = np.array_equal(ref, want)
    # B = I on the right (K = N): C = alpha*A + beta*C
    A2 = uniform(rng, M * K).reshape(M, K)
    B2 = np.eye(K, N, dtype=np.float32)
    ref2, _ = oracle.sgemm_ref(M, N, K, -4.0, A2, K, B2, N, 0.25, C, N, plant=plant)
    want2 = -4.0 * A2.astype(np.float64) + 0.25 * C.astype(np.float64)
    return ok_left and np.array_equal(ref2, want2)


def pin_permutation(plant=0) -> bool:
    """A = permutation matrix P: C = P @ B is B with rows permuted, exactly."""
    M = K = 29
    N = 41
    rng = np.random.default_rng(12)
    perm = rng.permutation(M)
    A = np.zeros((M, K), dtype=np.float32)
    A[np.arange(M), perm] = 1.0
    B = uniform(rng, K * N).reshape(K, N)
    ref, _ = oracle.sgemm_ref(M, N, K, 1.0, A, K, B, N, 0.0, None, N, plant=plant)
    return np.array_equal(ref, B[perm].astype(np.float64))


def pin_small_integers(plant=0) -> bool:
    """Integers in [-8, 8]: every sum is exact; compare with int64 matmul."""
    rng = np.random.default_rng(13)
    M, N, K = 45, 53, 67
    Ai = rng.integers(-8, 9, size=(M, K))
    Bi = rng.integers(-8, 9, size=(K, N))
    Ci = rng.integers(-8, 9, size=(M, N))
    A, B, C = (x.astype(np.float32) for x in (Ai, Bi, Ci))
    ref, scale = oracle.sgemm_ref(M, N, K, 3.0, A, K, B, N, -2.0, C, N, plant=plant)
    want = 3 * (Ai @ Bi) - 2 * Ci
    want_scale = 3 * (np.abs(Ai) @ np.abs(Bi)) + 2 * np.abs(Ci)
    return np.array_equal(ref, want.astype(np.float64)) and \
        np.array_equal(scale, want_scale.astype(np.float64))


def pin_constant_matrices(plant=0) -> bool:
    """The page's constant inputs (A = 1.0f, B = 0.01f, K = 1024): C = K*a*b."""
    with open(os.path.join(GOLDEN, "constant_matrices.json")) as f:
        g = json.load(f)
    a = np.float32(g["a"])
    b = np.float32(g["b"])
    K = int(g["K"])
    M, N = 16, 24        # the closed form holds for every M, N; keep it small
    A = np.full((M, K), a, dtype=np.float32)
    B = np.full((K, N), b, dtype=np.float32)
    ref, scale = oracle.sgemm_ref(M, N, K, 1.0, A, K, B, N, 0.0, None, N, plant=plant)
    exact = Fraction(K) * Fraction(float(a)) * Fraction(float(b))
    # the float64 running sum of K equal terms may round; allow K ulps
    tol = K * 2.0 ** -52 * float(exact)
    return bool(np.all(np.abs(ref - float(exact)) <= tol)) and \
        bool(np.all(np.abs(scale - float(exact)) <= tol))


def pin_alpha_beta_algebra(plant=0) -> bool:
    """sgemm(alpha, beta) = alpha * sgemm(1, 0) + beta * C (up to float64 rounding)."""
    p = random_problem(33, 47, 61, alpha=1.0, beta=0.0, seed=14)
    base, base_scale = oracle.sgemm_ref(p.M, p.N, p.K, 1.0, p.A, p.lda, p.B, p.ldb,
                                        0.0, None, p.ldc, plant=plant)
    Cv = p.C[:, :p.N].copy()
    Cv[:] = uniform(np.random.default_rng(15), p.M * p.N).reshape(p.M, p.N)
    alpha, beta = -1.75, 0.625
    ref, scale = oracle.sgemm_ref(p.M, p.N, p.K, alpha, p.A, p.lda, p.B, p.ldb,
                                  beta, Cv, p.N, plant=plant)
    want = alpha * base + beta * Cv.astype(np.float64)
    tol = 1e-14 * (abs(alpha) * base_scale + abs(beta) * np.abs(Cv))
    return bool(np.all(np.abs(ref - want) <= tol))


def pin_bruteforce_fractions(plant=0) -> bool:
    """Tiny random shapes against exact rational arithmetic."""
    rng = np.random.default_rng(16)
    for M, N, K in [(1, 1, 1), (2, 3, 4), (5, 4, 6), (6, 6, 6), (3, 1, 5)]:
        A = uniform(rng, M * K).reshape(M, K)
        B = uniform(rng, K * N).reshape(K, N)
        C = uniform(rng, M * N).reshape(M, N)
        alpha, beta = 1.25, -0.75
        ref, scale = oracle.sgemm_ref(M, N, K, alpha, A, K, B, N, beta, C, N, plant=plant)
        for m in range(M):
            for n in range(N):
                s = sum(Fraction(float(A[m, k])) * Fraction(float(B[k, n])) for k in range(K))
                t = sum(abs(Fraction(float(A[m, k])) * Fraction(float(B[k, n]))) for k in range(K))
                exact = Fraction(alpha) * s + Fraction(beta) * Fraction(float(C[m, n]))
                exact_scale = abs(Fraction(alpha)) * t + abs(Fraction(beta) * Fraction(float(C[m, n])))
                # K roundings of the running sum plus two in the epilogue
                tol = (K + 3) * 2.0 ** -53 * float(exact_scale)
                if abs(ref[m, n] - float(exact)) > tol:
                    return False
                if abs(scale[m, n] - float(exact_scale)) > tol:
                    return False
    return True


def pin_numpy_float64(plant=0) -> bool:
    """An independent float64 formulation (numpy matmul) at a few hundred."""
    p = random_problem(200, 176, 256, alpha=0.5, beta=2.0, seed=17, pad_value=0.0)
    p.C[:, :p.N] = uniform(np.random.default_rng(18), p.M * p.N).reshape(p.M, p.N)
    ref, scale = _ref(p, plant=plant)
    A = p.A[:, :p.K].astype(np.float64)
    B = p.B[:, :p.N].astype(np.float64)
    C = p.C[:, :p.N].astype(np.float64)
    want = p.alpha * (A @ B) + p.beta * C
    want_scale = abs(p.alpha) * (np.abs(A) @ np.abs(B)) + np.abs(p.beta * C)
    return bool(np.all(np.abs(ref - want) <= 1e-12 * want_scale)) and \
        bool(np.all(np.abs(scale - want_scale) <= 1e-12 * want_scale))


PINS = [pin_identity, pin_permutation, pin_small_integers, pin_constant_matrices,
        pin_alpha_beta_algebra, pin_bruteforce_fractions, pin_numpy_float64]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin_holds(oracle_mod, pin):
    assert pin(0), pin.__doc__


# ------------------------------------------------------- semantics readings

def test_beta_zero_does_not_read_c(oracle_mod):
    p = random_problem(17, 19, 23, beta=0.0, seed=21)
    p.C[:] = np.nan
    ref, scale = _ref(p)
    assert np.all(np.isfinite(ref)) and np.all(np.isfinite(scale))
    ref2, _ = oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb,
                               0.0, None, p.ldc)
    assert np.array_equal(ref, ref2)


@pytest.mark.parametrize("alpha,K", [(0.0, 23), (1.0, 0), (0.0, 0)])
def test_alpha_or_k_zero_does_not_read_ab(oracle_mod, alpha, K):
    M, N = 13, 11
    C = uniform(np.random.default_rng(22), M * N).reshape(M, N)
    A = np.full((M, max(K, 1)), np.nan, dtype=np.float32)
    B = np.full((max(K, 1), N), np.nan, dtype=np.float32)
    ref, scale = oracle.sgemm_ref(M, N, K, alpha, A, max(K, 1), B, N, 0.5, C, N)
    assert np.array_equal(ref, 0.5 * C.astype(np.float64))
    assert np.array_equal(scale, np.abs(0.5 * C.astype(np.float64)))
    ref0, _ = oracle.sgemm_ref(M, N, K, alpha, None, max(K, 1), None, N, 0.5, C, N)
    assert np.array_equal(ref, ref0)


def test_leading_dimension_padding(oracle_mod):
    """Padded lda/ldb/ldc (padding holds NaN) gives the packed result exactly."""
    M, N, K = 31, 45, 27
    packed = random_problem(M, N, K, 1.5, 0.5, seed=23, pad_value=0.0)
    packed.C[:, :N] = uniform(np.random.default_rng(24), M * N).reshape(M, N)
    padded = random_problem(M, N, K, 1.5, 0.5, seed=23, lda=K + 5, ldb=N + 3,
                            ldc=N + 7, pad_value=np.nan)
    padded.A[:, :K] = packed.A[:, :K]
    padded.B[:, :N] = packed.B[:, :N]
    padded.C[:, :N] = packed.C[:, :N]
    r1, s1 = _ref(packed)
    r2, s2 = _ref(padded)
    assert np.array_equal(r1, r2) and np.array_equal(s1, s2)


def test_row_sampling_matches_full(oracle_mod):
    p = random_problem(64, 40, 50, 1.0, 0.0, seed=25)
    full, fscale = _ref(p)
    rows = [0, 63, 17, 5, 17]
    part, pscale = _ref(p, rows=rows)
    assert np.array_equal(part, full[rows]) and np.array_equal(pscale, fscale[rows])


def test_special_values_follow_ieee_double(oracle_mod):
    M, N, K = 3, 4, 2
    A = np.array([[np.inf, 1.0], [np.nan, 1.0], [1.0, -1.0]], dtype=np.float32)
    B = np.array([[1.0, -2.0, 0.0, 1.0], [1.0, 1.0, 1.0, np.inf]], dtype=np.float32)
    ref, _ = oracle.sgemm_ref(M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    assert ref[0, 0] == np.inf and ref[0, 1] == -np.inf and np.isnan(ref[0, 2])
    assert np.all(np.isnan(ref[1]))
    assert ref[2, 0] == 0.0 and ref[2, 3] == -np.inf


def test_within_bound_rule():
    ref = np.array([1.0, -2.0, np.inf, np.nan, 0.0])
    scale = np.array([10.0, 10.0, np.inf, np.nan, 0.0])
    got = np.array([1.0 + 9e-4, -2.0 - 1.1e-3, np.inf, np.nan, 0.0])
    ok = oracle.within_bound(got, ref, scale)
    assert ok.tolist() == [True, False, True, True, True]
    assert not oracle.within_bound(np.array([np.nan]), np.array([1.0]), np.array([1.0]))[0]
    assert not oracle.within_bound(np.array([1e30]), np.array([np.inf]), np.array([np.inf]))[0]
    assert not oracle.within_bound(np.array([1e-30]), np.array([0.0]), np.array([0.0]))[0]


def test_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle.sgemm_ref(-1, 2, 2, 1.0, None, 2, None, 2, 0.0, None, 2)
    A = np.zeros((2, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.sgemm_ref(2, 2, 2, 1.0, A, 2, A, 2, 0.0, None, 2, rows=[2])


# ------------------------------------------------------ planted mistakes

@pytest.mark.parametrize("plant,what", [(1, "A read transposed"),
                                        (2, "beta term dropped"),
                                        (3, "last k dropped"),
                                        (4, "alpha and beta swapped")])
def test_each_planted_mistake_fails_a_pin(oracle_mod, plant, what):
    oracle.build(plant)
    failed = [p.__name__ for p in PINS if not p(plant)]
    assert failed, f"no pin catches the planted mistake: {what}"
