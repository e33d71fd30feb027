"""Host-side logic of bench.py that needs no GPU: the DRAM traffic reported
beside the roofline comes from the committed ncu record only while the
kernel source it was captured on is unchanged; the algorithmic work per
kernel, the roofline arithmetic and the CPU oracle legs."""
import hashlib
import json
import os

import pytest

import bench
from mixture_experts_ffn_softmax_gb300 import ncu_traffic
from mixture_experts_ffn_softmax_gb300 import workloads as wl


def _tree(tmp_path, src_text, rec):
    csrc = tmp_path / "pkg" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "gemm.cu").write_text(src_text)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic_gemm1_swiglu_wl.json").write_text(json.dumps(rec))


def _rec(sha, **kw):
    r = {"kernel": "gemm1_swiglu", "workload": "wl", "ncu_kernel": "k", "launch": 0,
         "dram_bytes_read": 12000, "dram_bytes_write": 345, "traffic_bytes_per_launch": 12345,
         "source": "pkg/csrc/gemm.cu", "source_sha256_16": sha, "command": "ncu ..."}
    r.update(kw)
    return r


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = "// kernel source\n"
    sha = hashlib.sha256(src.encode()).hexdigest()[:16]
    _tree(tmp_path, src, _rec(sha))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    v, note = bench.measured_traffic("gemm1_swiglu", "wl")
    assert v == 12345 and sha in note
    # another kernel or workload has no record
    assert bench.measured_traffic("gemm2_sorted", "wl")[0] is None
    # the source changed after the capture: no figure, and the line says why
    (tmp_path / "pkg" / "csrc" / "gemm.cu").write_text(src + " ")
    v, note = bench.measured_traffic("gemm1_swiglu", "wl")
    assert v is None and note.startswith("stale")


def test_traffic_record_must_match_its_name(tmp_path, monkeypatch):
    src = "x"
    sha = hashlib.sha256(src.encode()).hexdigest()[:16]
    _tree(tmp_path, src, _rec(sha, workload="other"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("gemm1_swiglu", "wl")[0] is None
    monkeypatch.setattr(bench, "ROOT", os.path.join(str(tmp_path), "missing"))
    assert bench.measured_traffic("gemm1_swiglu", "wl") == (None, "no ncu record")


def test_ncu_traffic_reads_both_export_forms(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("k")
    raw = ('==PROF== Connected\n'
           '"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum"\n'
           '"","","byte","Mbyte"\n'
           '"0","void other_kernel()","1","1"\n'
           '"1","void grouped_gemm_pair_kernel<0, 0>()","1953712896","231.77344"\n')
    rec = ncu_traffic.record(raw, "gemm1_swiglu", "wl", "grouped_gemm", 0, str(src), "cmd")
    assert rec["dram_bytes_read"] == 1953712896 and rec["dram_bytes_write"] == 231773440
    assert rec["traffic_bytes_per_launch"] == 1953712896 + 231773440
    assert rec["source_sha256_16"] == ncu_traffic.source_hash(str(src))
    long = ('"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
            '"3","grouped_gemm_kernel","dram__bytes_read.sum","byte","100"\n'
            '"3","grouped_gemm_kernel","dram__bytes_write.sum","byte","20"\n'
            '"4","grouped_gemm_kernel","dram__bytes_read.sum","Kbyte","1.5"\n'
            '"4","grouped_gemm_kernel","dram__bytes_write.sum","byte","7"\n')
    assert ncu_traffic.launches(long, "grouped") == [("grouped_gemm_kernel", 100, 20),
                                                    ("grouped_gemm_kernel", 1500, 7)]
    with pytest.raises(SystemExit):
        ncu_traffic.record(long, "g", "wl", "grouped", 5, str(src), "cmd")


def test_kernel_work_matches_the_layer_totals():
    """GEMM1 + GEMM2 FLOPs are the layer's 6 R H I; GEMM weight bytes are the
    touched experts' 3 H I bf16 values."""
    s = wl.SPECS["mixtral_prefill"]
    f1, b1 = bench.kernel_work("gemm1_swiglu", s.H, s.I, s.E, s.top_k, s.M, s.R, 8)
    f2, b2 = bench.kernel_work("gemm2_sorted", s.H, s.I, s.E, s.top_k, s.M, s.R, 8)
    assert f1 + f2 == s.flops()
    assert b1 == 8 * 4 * s.H * s.I + s.R * (2 * s.H + 2 * s.I)
    assert b2 == 8 * 2 * s.H * s.I + s.R * (2 * s.I + 4 * s.H)
    assert bench.kernel_work("reduce_sorted", s.H, s.I, s.E, 2, s.M, s.R, 8)[1] == \
        s.M * (8 * s.H + 2 * s.H)
    assert bench.kernel_work("no_such_kernel", 1, 1, 1, 1, 1, 1, 1) is None


def test_kernel_work_small_calls_and_gather():
    """The small-call GEMMs do the layer's 6 R H I FLOPs between them; their
    bytes are the touched experts' weights, the rows and z, plus the fp32
    token accumulator (zeroed by GEMM1, read back by GEMM2 with y written).
    The gather reads each token row once and writes each routed row once;
    the batched layout (M = R) reads and writes each row once."""
    s = wl.SPECS["tiny"]
    f1, b1 = bench.kernel_work("small_gemm1", s.H, s.I, s.E, s.top_k, s.M, s.R, 8)
    f2, b2 = bench.kernel_work("small_gemm2", s.H, s.I, s.E, s.top_k, s.M, s.R, 8)
    assert f1 + f2 == s.flops()
    assert b1 == 8 * 4 * s.H * s.I + s.R * (2 * s.H + 2 * s.I) + s.M * 4 * s.H
    assert b2 == 8 * 2 * s.H * s.I + s.R * 2 * s.I + s.M * 6 * s.H
    q = wl.SPECS["qwen_skew"]
    assert bench.kernel_work("gather_rows", q.H, q.I, q.E, q.top_k, q.M, q.R, 128)[1] == \
        q.M * 2 * q.H + q.R * 2 * q.H
    assert bench.kernel_work("gather_rows", q.H, q.I, q.E, 1, q.R, q.R, 128)[1] == q.R * 4 * q.H


def test_roofline_picks_the_binding_term():
    pk = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "hbm_gbs": 8000.0}
    # 2 TFLOP and 1 GB in 2 ms: tensor term 1 ms, HBM term 0.125 ms
    r = bench.roofline_of(2e12, 1e9, 2e-3, pk)
    assert r["bound"] == "tensor" and r["frac"] == 0.5 and r["achieved"] == 1000.0
    assert r["frac_of_sustained_peak"] == 0.625
    r = bench.roofline_of(1e9, 8e9, 2e-3, pk)
    assert r["bound"] == "hbm" and r["frac"] == 0.5 and r["achieved"] == 4000.0
    kern = {"a": {"launches": 1, "avg_us": 10.0}, "b": {"launches": 3, "avg_us": 5.0}}
    name, share, w = bench.dominant_kernel(kern, {"b": (1.0, 2.0)})
    assert name == "b" and share == 0.6 and w == (1.0, 2.0)


def test_cpu_baselines_run_on_a_sample():
    spec = wl.SPECS["tiny"]
    d = wl.make_moe_inputs(spec, device="cpu")
    r = bench.cpu_baseline(spec, d, budget_s=0.5)
    assert r["value"] > 0 and r["kind"] == "oracle" and "64 of 64 tokens" in r["sample"]
    bspec = wl.SMALL_BATCHED_SPECS["batched_small"]
    b = wl.make_batched_inputs(bspec, device="cpu")
    r = bench.cpu_baseline_batched(bspec, b, budget_s=0.5)
    assert r["value"] > 0 and "experts 0..1" in r["sample"]


def test_sample_bounds_the_widened_experts():
    for spec in wl.SPECS.values():
        n = bench._sample_tokens(spec)
        assert 1 <= n <= spec.M
        widened = min(spec.E, n * spec.top_k) * 3 * spec.H * spec.I * 8
        assert widened <= 12e9, spec.name
    assert bench._sample_tokens(wl.SPECS["deepseek_m8192"]) == 2
