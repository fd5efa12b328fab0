"""bench.py's roofline arithmetic, on the host: the algorithmic FLOPs and bytes of a forward (6·T·d·
(k·f + f_s) and 6·d·f·(E_act + S) + 4·T·d + 4·T·E) reproduce the figures worked out for the layer
shapes, the binding roof picks the larger of the tensor and HBM times, and a committed ncu
summary's traffic is used only while its kernel source is unchanged."""
import hashlib
import os

import pytest

import bench
from paged_moe_expert_gb300 import synthetic as syn


@pytest.mark.parametrize("name,T,e_act,gflop,mb", [
    ("qwen15", 1, 4, 0.138, 138.0),
    ("qwen15", 4096, 60, 567.0, 1141.0),
    ("mixtral", 8192, 8, 5772.0, 2953.0),
    ("qwen3next", 4096, 512, 283.0, 3261.0),
])
def test_algorithmic_work(name, T, e_act, gflop, mb):
    w = bench.work(syn.CONFIGS[name], T, e_act)
    assert w["flops"] / 1e9 == pytest.approx(gflop, rel=0.01)
    assert w["bytes"] / 1e6 == pytest.approx(mb, rel=0.01)
    # the two GEMMs split the FLOPs 2:1 and together carry every weight byte
    assert w["gemm1"]["flops"] + w["gemm2"]["flops"] == pytest.approx(w["flops"])
    assert w["gemm1"]["flops"] == pytest.approx(2 * w["gemm2"]["flops"])


def test_binding_fraction_takes_the_slower_roof():
    peaks = {"bf16_tflops_sustained": 1000.0, "bf16_tflops": 1200.0, "hbm_gbs": 5000.0}
    # 1 TFLOP at 1 PF/s = 1 ms; 1 GB at 5 TB/s = 0.2 ms: tensor-bound, measured 2 ms -> 0.5
    frac, bound = bench.binding_fraction(1e12, 1e9, 2e-3, peaks)
    assert bound == "tensor" and frac == pytest.approx(0.5)
    frac, bound = bench.binding_fraction(1e9, 1e10, 4e-3, peaks)
    assert bound == "hbm" and frac == pytest.approx(0.5)


def test_measured_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "paged_moe_expert_gb300" / "csrc"
    prof = tmp_path / "profiles"
    src.mkdir(parents=True)
    prof.mkdir()
    (src / "tc_gemm2sm.cu").write_text("// kernel v1\n")
    sha = hashlib.sha256(b"// kernel v1\n").hexdigest()[:16]
    (prof / "tc_gemm2sm_qwen15_T4096.md").write_text(
        "# summary\ntraffic_gemm1_bytes_per_launch: 123\ntraffic_source_sha256_prefix: %s\n" % sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("qwen15", 4096, "tc2", "gemm1") == 123
    assert bench.measured_traffic("qwen15", 4096, "tc2", "gemm2") is None      # not captured
    assert bench.measured_traffic("qwen15", 1024, "tc2", "gemm1") is None      # no summary
    (src / "tc_gemm2sm.cu").write_text("// kernel v2\n")
    assert bench.measured_traffic("qwen15", 4096, "tc2", "gemm1") is None      # stale


def test_job_throughput_counts_all_ranks():
    assert bench.job_throughput(100.0, 4, 2.0) == pytest.approx(200.0)


def test_dominant_kernel_takes_the_burst_peak_in_short_regions():
    peaks = {"bf16_tflops_sustained": 1000.0, "bf16_tflops": 1200.0, "hbm_gbs": 5000.0,
             "sm_max_mhz": 2000.0}
    kw = {"flops": 1.2e12, "bytes": 1e9}          # tensor-bound; 1 ms at the burst peak
    short = bench.dominant_roofline(kw, 2e-3, 4, peaks, region_s=0.1)
    assert short["bound"] == "tensor" and short["peak"] == 1200.0 and short["peak_kind"] == "burst"
    assert short["frac"] == pytest.approx(0.5)
    long = bench.dominant_roofline(kw, 2e-3, 4, peaks, region_s=2.5)
    assert long["peak"] == 1000.0 and long["peak_kind"] == "sustained"
    mem = bench.dominant_roofline({"flops": 1e9, "bytes": 1e10}, 4e-3, 5, peaks, region_s=0.1)
    assert mem["bound"] == "hbm" and mem["frac"] == pytest.approx(0.5)


def test_kernel_names_follow_the_launch_sequence():
    """The per-kernel timings are labelled from the launch count and the path: the routing kernel
    and the multi-CTA sort, or the one-CTA prep; a separate row gather on the tensor-core paths
    unless the prep copies the rows; one launch for the whole layer on the decode kernels."""
    ids = bench.PATH_IDS
    assert bench.kernel_names(6, ids["tc2"]) == ["route", "align", "gather", "gemm1", "gemm2", "combine"]
    assert bench.kernel_names(5, ids["tc_decode"]) == ["prep", "gather", "gemm1", "gemm2", "combine"]
    assert bench.kernel_names(5, ids["stream"]) == ["route", "align", "gemm1", "gemm2", "combine"]
    assert bench.kernel_names(4, ids["tc_decode"]) == ["prep", "gemm1", "gemm2", "combine"]
    assert bench.kernel_names(1, ids["fused"]) == ["fused"]
    assert bench.kernel_names(1, ids["slice"]) == ["fused"]
