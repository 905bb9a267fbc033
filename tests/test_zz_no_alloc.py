"""sgemm_noalloc: the entry point for callers that must not have the library
allocate device memory (a GPU fully reserved by the caller's own memory pool,
or a latency-sensitive loop that cannot absorb cudaMalloc's device-wide
synchronisation).  Its split-K scratch lives in a fixed array compiled into
the library.

Checked through the C ABI against the existing entry point (sgemm_ex with the
same path and split count) on two calls in a row, so that leftovers of the
first call in the shared array cannot leak into the second: both calls run
the same kernel on the same plan, so the results must be the same bits, and
both must pass the oracle's tolerance.  Also checked: after the documented
set-up call the device's free memory does not change across calls, and a
call whose bounded wait runs out (test hook) is reported by
sgemm_check_status, after which the next call is correct.  Collected last
(file name) so that a run stopping at the first failure has already run
everything else; it also passes alone in a fresh process.
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


def _setup_call(C, st):
    """The documented set-up call: alpha = 0, beta = 1 (C untouched)."""
    rc = pkg.sgemm_noalloc(1, 1, 0, 0.0, None, 1, None, 1, 1.0, C, 1, st, 0)
    assert rc == 0, pkg.sgemm_status_string(rc)


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
        assert torch.equal(C_noalloc, C_ex), f"call {call}: differs from sgemm_ex"
        got = C_noalloc.cpu().numpy()[:, :p.N].astype(np.float64)
        assert not oracle.first_failures(got, ref, scale), f"call {call}: differs from the oracle"


def test_noalloc_leaves_free_memory_unchanged():
    """After the set-up call, GEMMs of several plans (split-K, whole tiles,
    tensor-map and element-load operands, CTA pairs) take no device
    memory."""
    import torch
    st = torch.cuda.current_stream()
    cases = []
    for (M, N, K, off, splits) in [(1024, 1024, 1024, 0, 4), (333, 517, 301, 1, 2), (64, 4096, 147, 0, 1),
                                   (512, 384, 2048, 0, 0), (2560, 5120, 768, 0, 0)]:
        p = random_problem(M, N, K, alpha=1.0, beta=0.5, seed=M + N + K, pad_value=0.0)
        A = torch.zeros(p.A.size + 4, device="cuda")
        B = torch.zeros(p.B.size + 4, device="cuda")
        C = torch.zeros(p.C.size + 4, device="cuda")
        A[off:off + p.A.size] = torch.from_numpy(p.A.reshape(-1)).cuda()
        B[off:off + p.B.size] = torch.from_numpy(p.B.reshape(-1)).cuda()
        cases.append((p, A[off:], B[off:], C[off:], splits))
    _setup_call(cases[0][3], st)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        for p, A, B, C, splits in cases:
            rc = pkg.sgemm_noalloc(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, st, splits)
            assert rc == 0, pkg.sgemm_status_string(rc)
    assert pkg.sgemm_check_status(st) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes across sgemm_noalloc calls"


def test_noalloc_cta_pairs():
    """A plan on CTA pairs (256-row tiles): sgemm_noalloc matches the oracle
    on sampled rows and gives the same bits as sgemm_ex with the same
    schedule (whole tiles when the split tail's partial tiles would not fit
    sgemm_noalloc's 16 MiB of scratch, which then drops the tail)."""
    import torch
    M, N, K = 2560, 5120, 768
    p = random_problem(M, N, K, alpha=1.25, beta=0.5, seed=77, pad_value=0.0)
    p.C[:, :p.N] = uniform(np.random.default_rng(78), p.M * p.N).reshape(p.M, p.N)
    plan = pkg.sgemm_plan_info(M, N, K, algo=pkg.SGEMM_ALGO_TF32X3, beta=p.beta, num_sms=0)
    assert plan["pairs"] == 1, plan
    same_schedule = pkg.SGEMM_FLAG_WHOLE_TILES if plan["ws_bytes"] > (16 << 20) else 0
    st = torch.cuda.current_stream()
    A, B = torch.from_numpy(p.A).cuda(), torch.from_numpy(p.B).cuda()
    C1, C2 = torch.from_numpy(p.C).cuda(), torch.from_numpy(p.C).cuda()
    assert pkg.sgemm_noalloc(M, N, K, p.alpha, A, p.lda, B, p.ldb, p.beta, C1, p.ldc, st, 0) == 0
    assert pkg.sgemm_ex(M, N, K, p.alpha, A, p.lda, B, p.ldb, p.beta, C2, p.ldc, st, pkg.SGEMM_ALGO_TF32X3, 0,
                        same_schedule) == 0
    assert pkg.sgemm_check_status(st) == 0
    assert torch.equal(C1, C2)
    rows = [0, 255, 256, 1000, 2047, 2559]
    ref, scale = oracle.sgemm_ref(M, N, K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, p.C, p.ldc, rows=rows)
    assert not oracle.first_failures(C1.cpu().numpy()[rows, :N], ref, scale)


def test_noalloc_timeout_is_reported_and_cleared():
    """A call whose bounded wait runs out (the test hook withholds one
    pipeline arrive and cuts the budget to ~1 ms) sets sgemm_noalloc's status
    word; sgemm_check_status reports it and clears the word and the arrival
    counters, and the next split-K call is correct again."""
    import torch
    p = make_problem("square1024", pad_value=0.0)
    A, B, C0 = _device(p)
    st = torch.cuda.current_stream()
    assert pkg.sgemm_noalloc_debug_flags(pkg.SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE) == 0
    C = C0.clone()
    assert pkg.sgemm_noalloc(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, st, 4) == 0
    assert pkg.sgemm_check_status(st) == pkg.SGEMM_ERR_DEVICE_TIMEOUT
    assert pkg.sgemm_check_status(st) == 0  # read and cleared
    C = C0.clone()
    C_ex = C0.clone()
    assert pkg.sgemm_noalloc(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, st, 4) == 0
    assert pkg.sgemm_ex(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C_ex, p.ldc, st,
                        pkg.SGEMM_ALGO_TF32X3, 4, 0) == 0
    assert pkg.sgemm_check_status(st) == 0
    assert torch.equal(C, C_ex)
    assert pkg.sgemm_noalloc_debug_flags(2) == -1


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
