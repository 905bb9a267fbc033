"""sgemm_noalloc: the entry point for callers that must not have the library
allocate device memory (a GPU fully reserved by the caller's own memory pool,
or a latency-sensitive loop that cannot absorb cudaMalloc's device-wide
synchronisation).  Its split-K scratch lives in a fixed array compiled into
the library.

Checked through the C ABI against the existing entry point (sgemm_ex with the
same path and split count) with the parity tolerance of the other tests, on
two calls in a row, so that leftovers of the first call in the shared array
cannot leak into the second.  Collected last (file name) so that a run
stopping at the first failure has already run everything else; it also
passes alone in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest

import dense_fp32_matrix_05_gb300 as pkg
import oracle
from dense_fp32_matrix_05_gb300.workloads import make_problem, random_problem, uniform

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _device(p):
    import torch
    return (torch.from_numpy(p.A).cuda(), torch.from_numpy(p.B).cuda(),
            torch.from_numpy(p.C).cuda())


@pytest.mark.parametrize("name,splits", [("square1024", 4), ("ragged1023x1021x1025", 3)])
def test_noalloc_matches_sgemm_ex_twice(name, splits):
    import torch
    p = make_problem(name, pad_value=0.0)
    plan = pkg.sgemm_plan_info(p.M, p.N, p.K, algo=pkg.SGEMM_ALGO_TF32X3, splits=splits, num_sms=0)
    assert plan["splits"] == splits and plan["ws_bytes"] > 0  # the split-K scratch is really used
    ref, scale = oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, p.C, p.ldc)
    A, B, C0 = _device(p)
    st = torch.cuda.current_stream()
    for call in range(2):
        C_noalloc = C0.clone()
        C_ex = C0.clone()
        rc = pkg.sgemm_noalloc(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C_noalloc, p.ldc,
                               st, splits)
        assert rc == 0, pkg.sgemm_status_string(rc)
        rc = pkg.sgemm_ex(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C_ex, p.ldc, st,
                          pkg.SGEMM_ALGO_TF32X3, splits, 0)
        assert rc == 0, pkg.sgemm_status_string(rc)
        assert pkg.sgemm_check_status(st) == 0
        got = C_noalloc.cpu().numpy()[:, :p.N].astype(np.float64)
        want = C_ex.cpu().numpy()[:, :p.N].astype(np.float64)
        assert np.all(np.abs(got - want) <= oracle.REL_TOL * scale), f"call {call}: differs from sgemm_ex"
        assert not oracle.first_failures(got, ref, scale), f"call {call}: differs from the oracle"


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch
    # 2048^3 in 16 K slices needs 64 MiB of partial tiles, over the 16 MiB array
    M = N = K = 2048
    plan = pkg.sgemm_plan_info(M, N, K, algo=pkg.SGEMM_ALGO_TF32X3, splits=16, num_sms=0)
    assert plan["ws_bytes"] > (16 << 20)
    A = torch.zeros((M, K), device="cuda")
    B = torch.zeros((K, N), device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    rc = pkg.sgemm_noalloc(M, N, K, 1.0, A, K, B, N, 0.0, C, N, torch.cuda.current_stream(), 16)
    assert rc == pkg.SGEMM_ERR_SCRATCH_LIMIT
    assert "scratch" in pkg.sgemm_status_string(rc)
    torch.cuda.synchronize()
    assert bool(torch.all(C == 7.0)), "a rejected call must not touch C"


def test_noalloc_without_split_and_quick_returns():
    import torch
    p = random_problem(300, 200, 150, alpha=1.5, beta=0.5, seed=41, pad_value=0.0)
    p.C[:, :p.N] = uniform(np.random.default_rng(42), p.M * p.N).reshape(p.M, p.N)
    ref, scale = oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, p.C, p.ldc)
    A, B, C = _device(p)
    st = torch.cuda.current_stream()
    assert pkg.sgemm_noalloc(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, st, 1) == 0
    assert not oracle.first_failures(C.cpu().numpy()[:, :p.N], ref, scale)
    # alpha == 0: C = beta * C, A and B not read
    C2 = C.clone()
    assert pkg.sgemm_noalloc(p.M, p.N, p.K, 0.0, None, p.lda, None, p.ldb, 2.0, C2, p.ldc, st, 0) == 0
    assert torch.equal(C2, 2.0 * C)
    # argument errors use the same numbering as sgemm_ex
    assert pkg.sgemm_noalloc(-1, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 4, st, 0) == -1
    assert pkg.sgemm_noalloc(4, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 4, st, -1) == -14
