"""bench.py host helpers on CPU: which measured peak a timed region is compared with, and the
DRAM-traffic lookup that is valid only while a kernel's sources are unchanged."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_long_loops_use_the_sustained_peak():
    assert bench.tensor_peak_key(750.0) == "bf16_tflops_sustained"
    assert bench.tensor_peak_key(500.0) == "bf16_tflops_sustained"
    assert bench.tensor_peak_key(232.0) == "bf16_tflops"
    peaks, _ = bench.measured_peaks()
    assert bench.tensor_peak_key(0.0) in peaks and bench.tensor_peak_key(1e4) in peaks


def test_every_kernel_has_its_own_source_hash():
    hashes = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert set(hashes) >= {"gsr_pair_kernel", "gsr_skinny_kernel", "gsr_tiled_kernel", "gsr_attention_kernel"}
    assert len(set(hashes.values())) == len(hashes)
    for k, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "tensor_core_gemm_multistage_gb300", f)), f


def test_traffic_is_reported_only_for_the_profiled_sources(tmp_path, monkeypatch):
    cur = bench.kernel_source_hash("gsr_pair_kernel")
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\nsquare8192 gsr_pair_kernel %s 123456 note\n"
                 "square8192 gsr_skinny_kernel %s 999 other kernel\n"
                 "llm_mlp_up gsr_pair_kernel 0000000000000000 777 stale\n" % (cur, cur))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.read_traffic("square8192", "gsr_pair_kernel") == 123456.0
    assert bench.read_traffic("llm_mlp_up", "gsr_pair_kernel") is None        # stale hash
    assert bench.read_traffic("skinny_decode", "gsr_pair_kernel") is None     # no line
    assert bench.read_traffic("square8192", "gsr_skinny_kernel") is None      # other kernel's hash


def test_source_hash_ignores_comments_but_not_code():
    code = "int f(int x) {\n    return x + 1;  // add one\n}\n/* block\n comment */\n"
    assert bench._code_only(code) == bench._code_only("int f(int x) { return x + 1; }")
    assert bench._code_only(code) != bench._code_only("int f(int x) { return x + 2; }")


def test_gemm_roofline_bounds_and_fractions():
    from tensor_core_gemm_multistage_gb300.workloads import WORKLOADS
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    w = WORKLOADS["llm_mlp_up"]
    r = bench.gemm_roofline(w, 2, "gsr_pair_kernel", 1.0, 20.0, peaks, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - w.flops / 1e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 1900.0) < 1e-12            # a 20 ms region: burst peak
    r = bench.gemm_roofline(w, 2, "gsr_pair_kernel", 1.0, 800.0, peaks, "measured")
    assert r["peak"] == 1700.0                                        # >= 0.5 s: sustained peak
    s = WORKLOADS["skinny_decode"]
    r = bench.gemm_roofline(s, 1, "gsr_skinny_kernel", 0.08, 16.0, peaks, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - s.bytes / 0.08e-3 / 1e9) < 1e-6 and abs(r["frac"] - r["achieved"] / 6800.0) < 1e-12


def test_per_config_entry_fields():
    from tensor_core_gemm_multistage_gb300.workloads import WORKLOADS
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    w = WORKLOADS["skinny_decode"]
    rec = {"step_ms": 0.1, "kernel_ms": 0.08, "median5_ms": 0.09, "region_ms": 2.0, "l2": "x"}
    e = bench.per_config_entry(w, rec, 1, "gsr_skinny_kernel", peaks, "measured", 1)
    assert e["kernel"] == "gsr_skinny_kernel" and e["ms_per_step"] == 0.1
    assert abs(e["TFLOP/s"] - w.flops / 0.1e-3 / 1e12) < 1e-9
    assert abs(e["median5_TFLOP/s"] - w.flops / 0.09e-3 / 1e12) < 1e-9
    assert abs(e["GB/s"] - w.bytes / 0.08e-3 / 1e9) < 1e-6
    assert e["roofline"]["bound"] == "hbm"
    assert "l2_warm" not in e                       # timed back to back already
    w1 = WORKLOADS["square1024"]                      # flushed: the warm figure rides along
    rec1 = dict(rec, warm_ms=0.01)
    e1 = bench.per_config_entry(w1, rec1, 0, "gsr_tiled_kernel", peaks, "measured", 1)
    assert abs(e1["l2_warm"]["TFLOP/s"] - w1.flops / 0.01e-3 / 1e12) < 1e-9
    assert "no flush" in e1["l2_warm"]["how"]


def test_host_cpu_model_is_a_string():
    m = bench.host_cpu_model()
    assert isinstance(m, str) and m


def test_oracle_baseline_full_and_sampled():
    from tensor_core_gemm_multistage_gb300.workloads import Workload, make_inputs
    w = Workload("t", 96, 64, 64, 0.5)
    A, B = make_inputs(w.M, w.N, w.K, seed=1)
    full = bench.oracle_baseline(A, B, w, 30.0)
    assert full["kind"] == "oracle" and "full_s" in full and full["sample"].startswith("all 96 rows")
    sampled = bench.oracle_baseline(A, B, w, 0.0)        # no time for all rows: a labelled sample
    assert "extrapolated_full_s" in sampled and "extrapolated" in sampled["extrapolated_note"]
    assert sampled["per_row_ms"] > 0 and sampled["value"] > 0


def test_clock_summary_windows_and_reasons():
    s = bench.ClockSampler("GPU-a")
    idle = ["Not Active"] * 5
    capped = ["Active", "Not Active", "Not Active", "Not Active", "Active"]
    s.samples = [(10.00, 2070.0, 2070.0, idle, "GPU-a"),
                 (10.02, 1980.0, 2070.0, capped, "GPU-a"),
                 (10.04, 2010.0, 2070.0, idle, "GPU-a"),
                 (10.02, 900.0, 2070.0, idle, "GPU-b")]       # another GPU's line
    got = s.summary(10.01, 10.05)
    assert got["samples"] == 2 and got["window"] == "timed region"
    assert got["sm_mhz"] == 1995.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]
    # a window between two samples falls back to the samples around it
    near = s.summary(10.041, 10.045)
    assert near["window"] == "around the timed region" and near["samples"] == 3
    assert bench.ClockSampler("GPU-x").summary(0, 1)["samples"] == 0
