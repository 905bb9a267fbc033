"""Host logic of bench.py that needs no GPU: which committed ncu summary a
bench line takes its DRAM traffic from, and when it takes none."""
import os

import pytest

import bench


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda family="tf32x3": "feedc0de12345678")
    return tmp_path


def _summary(root, name, hash_, nbytes):
    (root / "profiles" / f"{name}.md").write_text(
        f"# summary\n\nkernel_source_hash: {hash_}\ndram_bytes_per_launch: {nbytes}\n\ntext\n")


def test_traffic_comes_from_a_summary_of_the_current_sources(fake_root):
    _summary(fake_root, "tf32x3_square5120", "feedc0de12345678", 886701824)
    assert bench.recorded_traffic("square5120", "tf32x3") == 886701824.0
    assert bench.recorded_traffic("square1024", "tf32x3") is None          # no summary
    _summary(fake_root, "ffma_square5120", "0123456789abcdef", 1000789504)
    assert bench.recorded_traffic("square5120", "ffma") is None            # taken on other sources


def test_transposed_forms_use_their_own_summary(fake_root):
    _summary(fake_root, "tf32x3_square5120", "feedc0de12345678", 886701824)
    assert bench.profile_name("tf32x3") == "tf32x3"
    assert bench.profile_name("tf32x3", "NT") == "tf32x3_NT"
    assert bench.recorded_traffic("square5120", bench.profile_name("tf32x3", "TN")) is None
    _summary(fake_root, "tf32x3_NT_square5120", "feedc0de12345678", 887937024)
    assert bench.recorded_traffic("square5120", bench.profile_name("tf32x3", "NT")) == 887937024.0


def test_committed_summaries_name_their_sources_and_traffic():
    """Every committed summary records the source hash and the DRAM bytes
    per launch it was taken with, in the form the lookup reads."""
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles")
    names = [n for n in os.listdir(root) if n.endswith(".md")]
    assert names
    for n in names:
        text = open(os.path.join(root, n)).read()
        assert "kernel_source_hash:" in text and "dram_bytes_per_launch:" in text, n
        assert "--clock-control none" in text, n


def test_each_kernel_family_has_its_own_hash():
    """A summary is retired only by changes to its own kernel family's
    sources: the families hash different files."""
    assert bench.kernel_family("tf32x3_NT") == "tf32x3"
    assert bench.kernel_family("ffma_wide") == "ffma_wide"
    assert bench.kernel_family("ffma") == "ffma"
    hashes = {f: bench.kernel_source_hash(f) for f in bench.KERNEL_SOURCES}
    assert len(set(hashes.values())) == len(hashes)


def test_per_shape_summary_keeps_the_figures_and_the_l2_mode():
    gemm = {"config": {"workload": "square1024: M=1024 N=1024 K=1024 ...", "algo": "auto -> tf32x3",
                       "l2": "flushed between steps (512 MB written, untimed; ...)"},
            "value": 73.4, "unit": "TFLOP/s", "steps": 200,
            "roofline": {"bound": "tensor", "frac": 0.23, "launch_ms": 0.0293, "frac_of_mma_rate": 0.18},
            "clocks": {"sm_mhz": 2070.0, "reasons": []},
            "context_cublas_sgemm_tflops": 49.3,
            "context_back_to_back_l2_resident": {"value": 91.4}}
    s = bench.shape_summary(gemm)
    assert s["workload"] == "square1024" and s["l2"] == "flushed"
    assert (s["value"], s["frac"], s["frac_of_mma_rate"]) == (73.4, 0.23, 0.18)
    assert s["context_back_to_back_l2_resident"] == 91.4
    big = dict(gemm, config=dict(gemm["config"], l2="no flush: inputs larger than L2 (419 MB vs 129 MB)"))
    assert bench.shape_summary(big)["l2"] == "larger than L2"
    err = {"workload": "square256", "algo": "auto", "error": "boom"}
    assert bench.shape_summary(err) == err


def test_pipeline_bound_is_the_larger_of_the_copy_floor_and_prefix_plus_gemm():
    copy = {"h2d_gbs": 200.0, "copy_bound_ms": 1.5}
    # link-bound: 100 MB prefix (0.5 ms) + 0.8 ms GEMM is under the 1.5 ms copy floor
    b = bench.pipeline_bound(copy, 100e6, 0.8, 1.875)
    assert b["pipeline_bound_ms"] == 1.5 and b["frac_of_pipeline_bound"] == 0.8
    # GEMM-bound: 0.5 ms prefix + 24 ms GEMM
    b = bench.pipeline_bound(copy, 100e6, 24.0, 30.625)
    assert b["pipeline_bound_ms"] == 24.5 and b["frac_of_pipeline_bound"] == 0.8
