"""Host-side logic of bench.py that needs no GPU: the DRAM traffic reported
beside the roofline comes from the committed ncu summary only while the
kernel source it was captured on is unchanged."""
import hashlib
import os

import bench


def _tree(tmp_path, src_text, summary_text):
    csrc = tmp_path / "mixture_experts_ffn_softmax_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "gemm.cu").write_text(src_text)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "gemm_wl_ncu_full.md").write_text(summary_text)


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = "// kernel source\n"
    sha = hashlib.sha256(src.encode()).hexdigest()[:16]
    _tree(tmp_path, src, f"Source: csrc/gemm.cu sha256[:16] = {sha}\n"
                         "traffic_bytes_per_launch gemm1_swiglu wl: 12345\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("gemm1_swiglu", "wl") == 12345
    # another kernel or workload has no figure
    assert bench.measured_traffic("gemm2_sorted", "wl") is None
    # the source changed after the capture: no figure
    (tmp_path / "mixture_experts_ffn_softmax_gb300" / "csrc" / "gemm.cu").write_text(src + " ")
    assert bench.measured_traffic("gemm1_swiglu", "wl") is None


def test_traffic_needs_hash_and_figure(tmp_path, monkeypatch):
    _tree(tmp_path, "x", "traffic_bytes_per_launch gemm1_swiglu wl: 7\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("gemm1_swiglu", "wl") is None
    monkeypatch.setattr(bench, "ROOT", os.path.join(str(tmp_path), "missing"))
    assert bench.measured_traffic("gemm1_swiglu", "wl") is None
