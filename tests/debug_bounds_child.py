"""Runs in a child process of tests/test_zy_debug_bounds_gpu.py: loads the
SGEMM_DEBUG build of the library (every computed global address of the
kernels checked against its matrix, violations reported as
SGEMM_ERR_OUT_OF_BOUNDS; tensor maps that could reach outside their operand
refused) and runs parity cases that cross every tile edge, odd leading
dimensions, misaligned pointers, the residue-class form, CTA pairs, split-K
and split tails, the wide-N kernel, transposed operands, a strided batch,
convolutions and sgemm_noalloc.  Each must report status 0 and match the
float64 oracle.  Prints one line per case group; exits non-zero on failure."""
from __future__ import annotations

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import dense_fp32_matrix_05_gb300 as pkg  # noqa: E402
from dense_fp32_matrix_05_gb300 import _build_ext  # noqa: E402

DEBUG_LIB = _build_ext.build(debug=True)
pkg.lib_path = lambda: DEBUG_LIB  # this process uses the SGEMM_DEBUG build only

import oracle  # noqa: E402
from dense_fp32_matrix_05_gb300.workloads import random_problem, uniform  # noqa: E402
from gpu_util import check_against_oracle, run_sgemm  # noqa: E402


def with_c(p, seed):
    if p.beta != 0:
        p.C[:, :p.N] = uniform(np.random.default_rng(seed), p.M * p.N).reshape(p.M, p.N)
    return p


def gemm_cases():
    n = 0
    shapes = [(1, 1, 1), (7, 9, 5), (17, 15, 33), (63, 65, 64), (127, 129, 31), (129, 127, 65), (257, 130, 160),
              (33, 515, 20), (300, 1, 40), (1, 300, 40)]
    layouts = [((0, 0, 0), (0, 0, 0)), ((1, 3, 5), (0, 0, 0)), ((0, 0, 0), (1, 3, 2)), ((3, 1, 7), (2, 1, 3))]
    for algo in (pkg.SGEMM_ALGO_TF32X3, pkg.SGEMM_ALGO_FFMA):
        for M, N, K in shapes:
            for ld, off in layouts:
                p = with_c(random_problem(M, N, K, alpha=1.5, beta=0.5, seed=M + N + K, lda=K + ld[0],
                                          ldb=N + ld[1], ldc=N + ld[2]), 5)
                C, st = run_sgemm(p, algo, offsets=off)
                assert C is not None and st == 0, (M, N, K, ld, off, algo, st, pkg.sgemm_status_string(st))
                check_against_oracle(p, C, what=f"debug {M}x{N}x{K} ld+{ld} off{off} algo {algo}")
                n += 1
    # schedules and forms: split-K, split tail, whole tiles, tile heights,
    # residue-class B, staged A, B rows loaded, no A copy
    forms = [(300, 1021, 700, 0, pkg.SGEMM_FLAG_TILE_ROWS(128)), (384, 1413, 300, 3, pkg.SGEMM_FLAG_TILE_ROWS(192)),
             (130, 517, 37, 2, pkg.SGEMM_FLAG_TILE_ROWS(256)), (65, 265, 5, 0, pkg.SGEMM_FLAG_TILE_ROWS(64)),
             (64, 5000, 147, 1, 0), (32, 4100, 27, 2, pkg.SGEMM_FLAG_TILE_ROWS(32)),
             (300, 1021, 700, 0, pkg.SGEMM_FLAG_B_ROWS_LOADED), (40, 2000, 147, 0, pkg.SGEMM_FLAG_NO_A_COPY),
             (1000, 1000, 600, 0, pkg.SGEMM_FLAG_SPLIT_TAIL), (1000, 1000, 600, 0, pkg.SGEMM_FLAG_WHOLE_TILES)]
    # CTA pairs (A rows 16-byte aligned: K a multiple of 4): whole tiles with
    # ragged edges, residue-class B, 192-row tiles, forced split-K, and a
    # split tail over more tiles than pairs
    P = pkg.SGEMM_FLAG_PAIRS
    forms += [(300, 1021, 700, 0, pkg.SGEMM_FLAG_TILE_ROWS(256) | P | pkg.SGEMM_FLAG_WHOLE_TILES),
              (384, 1413, 300, 0, pkg.SGEMM_FLAG_TILE_ROWS(192) | P), (257, 129, 36, 3, pkg.SGEMM_FLAG_TILE_ROWS(256) | P),
              (1280, 4352, 256, 0, pkg.SGEMM_FLAG_TILE_ROWS(256) | P | pkg.SGEMM_FLAG_SPLIT_TAIL)]
    for M, N, K, splits, flags in forms:
        p = with_c(random_problem(M, N, K, alpha=0.75, beta=0.5, seed=M * 3 + K, pad_value=0.0), 6)
        C, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=splits, flags=flags)
        assert C is not None and st == 0, (M, N, K, splits, flags, st, pkg.sgemm_status_string(st))
        check_against_oracle(p, C, what=f"debug {M}x{N}x{K} splits {splits} flags {flags:#x}")
        n += 1
    # the wide-N FFMA kernel (AUTO for M <= 32, K <= 48), aligned and not
    for M, N, K, ldb in ((24, 1500, 27, 1500), (32, 3001, 40, 3003)):
        p = random_problem(M, N, K, alpha=-0.5, beta=0.0, seed=9, ldb=ldb, pad_value=0.0)
        C, st = run_sgemm(p, pkg.SGEMM_ALGO_AUTO)
        assert C is not None and st == 0, (M, N, K, st)
        check_against_oracle(p, C, what=f"debug wide {M}x{N}x{K}")
        n += 1
    return n


def other_entry_points():
    import torch
    st = torch.cuda.current_stream()
    n = 0
    # transposed operands: NT (B^T read in place), TN and TT (copies)
    M, N, K = 150, 260, 131
    p = random_problem(M, N, K, alpha=1.0, beta=0.5, seed=11, pad_value=0.0)
    p.C[:, :N] = uniform(np.random.default_rng(12), M * N).reshape(M, N)
    ref, scale = oracle.sgemm_ref(M, N, K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, p.C, p.ldc)
    for ta in (0, 1):
        for tb in (0, 1):
            A = torch.from_numpy(np.ascontiguousarray(p.A[:, :K].T) if ta else p.A).cuda()
            B = torch.from_numpy(np.ascontiguousarray(p.B[:, :N].T) if tb else p.B).cuda()
            C = torch.from_numpy(p.C).cuda()
            rc = pkg.sgemm_t(ta, tb, M, N, K, p.alpha, A, M if ta else p.lda, B, K if tb else p.ldb, p.beta, C,
                             p.ldc, st)
            status = pkg.sgemm_check_status(st)
            assert rc == 0 and status == 0, (ta, tb, rc, status)
            assert not oracle.first_failures(C.cpu().numpy()[:, :N], ref, scale), (ta, tb)
            n += 1
    # a strided batch with a shared A, one launch
    bs = [random_problem(96, 161, 48, alpha=1.0, beta=0.0, seed=20 + b, pad_value=0.0) for b in range(3)]
    A = torch.from_numpy(bs[0].A).cuda()
    B = torch.from_numpy(np.stack([b.B for b in bs])).cuda()
    C = torch.zeros((3, 96, 161), device="cuda")
    rc = pkg.sgemm_strided_batched(0, 0, 96, 161, 48, 1.0, A, 48, 0, B, 161, 48 * 161, 0.0, C, 161, 96 * 161, 3,
                                   st)
    status = pkg.sgemm_check_status(st)
    assert rc == 0 and status == 0, (rc, status)
    for b in range(3):
        r, s = oracle.sgemm_ref(96, 161, 48, 1.0, bs[0].A, 48, bs[b].B, 161, 0.0, None, 161)
        assert not oracle.first_failures(C[b].cpu().numpy(), r, s), b
    n += 1
    # convolutions: tap table with a zero-bordered copy, the bounds-checked
    # tap walk, channels order, and the wide FFMA form
    rng = np.random.default_rng(13)
    for C_in, F, pad, flags in ((3, 40, 1, 0), (3, 40, 1, pkg.SGEMM_CONV_NO_PAD_COPY), (16, 40, 1, 0),
                                (3, 8, 1, 0)):
        X = rng.random((2, C_in, 13, 15), dtype=np.float32) * 2 - 1
        Wt = rng.random((F, C_in, 3, 3), dtype=np.float32) * 2 - 1
        Y = torch.zeros((2, F, 13, 15), device="cuda")
        rc = pkg.sgemm_conv2d(torch.from_numpy(X).cuda(), torch.from_numpy(Wt).cuda(), Y, pad=(pad, pad),
                              stream=st, flags=flags)
        status = pkg.sgemm_check_status(st)
        assert rc == 0 and status == 0, (C_in, F, flags, rc, status)
        r, s = oracle.conv2d_ref(1.0, X, Wt, pad=(pad, pad))
        assert not oracle.first_failures(Y.cpu().numpy(), r, s), (C_in, F, flags)
        n += 1
    # sgemm_noalloc, split-K
    p = random_problem(512, 384, 700, alpha=1.0, beta=0.5, seed=14, pad_value=0.0)
    p.C[:, :] = uniform(np.random.default_rng(15), p.C.size).reshape(p.C.shape)
    ref, scale = oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, p.C, p.ldc)
    A, B, C = (torch.from_numpy(x).cuda() for x in (p.A, p.B, p.C))
    rc = pkg.sgemm_noalloc(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, st, 3)
    status = pkg.sgemm_check_status(st)
    assert rc == 0 and status == 0, (rc, status)
    assert not oracle.first_failures(C.cpu().numpy(), ref, scale)
    n += 1
    return n


def main():
    import torch
    torch.cuda.set_device(0)
    oracle.build()
    assert os.path.samefile(pkg.library()._name, DEBUG_LIB)
    print(f"debug build: {gemm_cases()} GEMM cases, {other_entry_points()} other calls, status 0 and oracle parity",
          flush=True)


if __name__ == "__main__":
    main()
