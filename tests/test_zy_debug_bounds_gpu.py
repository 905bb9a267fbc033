"""The SGEMM_DEBUG build as an out-of-bounds detector (compute-sanitizer is
not available here): every computed global address of the GEMM, FFMA,
wide-N and convolution kernels is checked against the byte range of its
matrix, a violation is skipped and reported (SGEMM_ERR_OUT_OF_BOUNDS from
sgemm_check_status, never a trap), and a tensor map that could reach outside
its operand is refused on the host.  The parity cases run in a child
process that loads that build (tests/debug_bounds_child.py), so this
process keeps the release library; they must all report status 0 and match
the oracle."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_finds_no_out_of_bounds_access():
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_child.py")], capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, f"stdout:\n{r.stdout[-3000:]}\nstderr:\n{r.stderr[-3000:]}"
    assert "status 0 and oracle parity" in r.stdout


def test_release_build_has_no_bounds_checks():
    """The checks compile away in the release build: its library and the
    debug one are different files, and only the debug one is built with
    SGEMM_DEBUG."""
    from dense_fp32_matrix_05_gb300 import _build_ext
    assert _build_ext.lib_path() != _build_ext.lib_path(debug=True)
    assert "-DSGEMM_DEBUG" not in _build_ext.CUDA_FLAGS
