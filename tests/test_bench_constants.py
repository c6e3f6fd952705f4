"""The bench's "of the pages' peak" denominators are the dense per-GPU figures
the pages print for HGX B200, stored with their citation under tests/golden/."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _golden(name):
    vals = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, value = line.split()
                vals[key] = float(value)
    return vals


def test_pages_peaks_match_the_spec_table():
    sys.path.insert(0, ROOT)
    import bench
    g = _golden("hgx_b200_dense_peaks.txt")
    assert bench.PAGES_PEAK_TFLOPS == {"bf16": g["bf16"] * 1000, "mxfp8": g["fp8"] * 1000,
                                       "nvfp4": g["nvfp4"] * 1000}
    assert bench.PAGES_HBM_GBS == g["hbm_tbs"] * 1000


def test_cpu_oracle_sweep_small_configs():
    # the bench's per-configuration oracle timing, on small shapes of each format
    sys.path.insert(0, ROOT)
    import bench
    out = bench.cpu_oracle_sweep([("bf16", "bf16", 64, 48, 64, 1, 64), ("mxfp8", "mxfp8", 32, 40, 64, 2, 16),
                                  ("nvfp4", "nvfp4", 32, 40, 64, 3, 8)])
    assert set(out) == {"bf16", "mxfp8", "nvfp4"}
    for label, rows in (("bf16", 64), ("mxfp8", 16), ("nvfp4", 8)):
        assert out[label]["rows"] == rows and out[label]["gflops"] > 0 and out[label]["seconds"] > 0


def test_kernel_hash_ignores_comments_only():
    # recorded counters stay valid across comment edits, not across code edits
    sys.path.insert(0, ROOT)
    import bench
    a = "int f() { return 1; }  // one\n/* a block\n   comment */\n\nint g();\n"
    b = "int f() { return 1; }  // other words\n\nint g();\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(a.replace("return 1", "return 2"))


def test_recorded_traffic_needs_the_current_kernel_hash(monkeypatch, tmp_path):
    # roofline.traffic comes from a capture only while the kernel sources are the captured ones
    import json
    sys.path.insert(0, ROOT)
    import bench
    rec = {"BF16 GEMM M=N=K=16384": {"dram_bytes_per_launch": 123.0, "kernel_hash": "abc"}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda: "abc")
    assert bench.recorded_traffic("BF16 GEMM M=N=K=16384") == 123.0
    assert bench.recorded_traffic("NVFP4 GEMM M=N=K=16384") is None
    monkeypatch.setattr(bench, "kernel_hash", lambda: "def")
    assert bench.recorded_traffic("BF16 GEMM M=N=K=16384") is None
