"""Helpers for the GPU parity tests: run one SGEMM through the C ABI on
device buffers surrounded by guard bands, and compare with the oracle."""
from __future__ import annotations

import numpy as np

import dense_fp32_matrix_05_gb300 as pkg
import oracle

GUARD = 1024          # floats of sentinel on each side of every device matrix
SENTINEL = np.float32(-1.2345678e30)


def _device_copy(host: np.ndarray, offset: int = 0):
    """Copy `host` to the device inside a guarded buffer.

    Returns (buffer, view) where view starts `offset` floats past a 256-byte
    aligned position (offset 1 gives a pointer that is not 16-byte aligned).
    """
    import torch
    flat = np.ascontiguousarray(host).reshape(-1)
    total = GUARD + offset + flat.size + GUARD
    buf = torch.full((total,), float(SENTINEL), dtype=torch.float32, device="cuda")
    start = GUARD + offset
    buf[start:start + flat.size] = torch.from_numpy(flat).to("cuda")
    return buf, start


def run_sgemm(p, algo=pkg.SGEMM_ALGO_AUTO, splits=0, offsets=(0, 0, 0), flags=0, stream=None):
    """Run C = alpha*A*B + beta*C for workload problem `p` on the GPU.

    Returns (C_host, status) where C_host has p.C's shape (ld columns).  Asserts
    that the guard bands around A, B and C are untouched and that A, B are not
    modified.
    """
    import torch
    bufA, sA = _device_copy(p.A, offsets[0])
    bufB, sB = _device_copy(p.B, offsets[1])
    bufC, sC = _device_copy(p.C, offsets[2])
    st = stream if stream is not None else torch.cuda.current_stream()
    esz = 4
    rc = pkg.sgemm_ex(p.M, p.N, p.K, p.alpha, bufA.data_ptr() + sA * esz, p.lda,
                      bufB.data_ptr() + sB * esz, p.ldb, p.beta, bufC.data_ptr() + sC * esz, p.ldc,
                      st, algo, splits, flags)
    if rc != 0:
        return None, rc
    status = pkg.sgemm_check_status(st)
    C = bufC.cpu().numpy()
    A = bufA.cpu().numpy()
    B = bufB.cpu().numpy()
    for name, arr, start, host in (("A", A, sA, p.A), ("B", B, sB, p.B), ("C", C, sC, p.C)):
        n = host.size
        assert np.all(arr[:start] == SENTINEL), f"write before {name}"
        assert np.all(arr[start + n:] == SENTINEL), f"write after {name}"
    assert np.array_equal(A[sA:sA + p.A.size].view(np.uint32), p.A.reshape(-1).view(np.uint32)), "A modified"
    assert np.array_equal(B[sB:sB + p.B.size].view(np.uint32), p.B.reshape(-1).view(np.uint32)), "B modified"
    return C[sC:sC + p.C.size].reshape(p.C.shape), status


def check_against_oracle(p, Cgot, rows=None, what=""):
    """Parity rule on all rows (or the sampled rows), plus untouched ld padding."""
    ref, scale = oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta,
                                  p.C if p.beta != 0 else None, p.ldc, rows=rows)
    got = Cgot[:, :p.N] if rows is None else Cgot[np.asarray(rows), :p.N]
    msg = oracle.first_failures(got, ref, scale)
    assert not msg, f"{what}: {msg}"
    if p.ldc > p.N:
        pad_got = Cgot[:, p.N:].view(np.uint32)
        pad_init = p.C[:, p.N:].view(np.uint32)
        assert np.array_equal(pad_got, pad_init), f"{what}: C padding columns modified"


def sample_rows(M: int, count: int = 64, seed: int = 0):
    if M <= count:
        return list(range(M))
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=count - 2, replace=False)
    return sorted({0, M - 1, *mid.tolist()})
