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
