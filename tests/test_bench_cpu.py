"""bench.py on the CPU: it imports, its entry points and helpers exist, the
recorded DRAM traffic table is well formed, and its source hash ignores
comments but not code."""
import importlib.util
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_entry_points_exist(bench):
    for name in ("main", "run_gb300", "run_prefill", "run_prefix_cache", "run_swap", "run_reference",
                 "cpu_baseline", "ClockSampler", "Batch", "Staging", "_source_sha", "_p10_p90"):
        assert hasattr(bench, name), name


def test_help_runs():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True,
                         text=True, timeout=120)
    assert out.returncode == 0 and "--workload" in out.stdout


def test_traffic_table_shape(bench):
    t = bench.NCU_TRAFFIC
    assert len(t["source_sha256"]) == 64
    for name, nbytes in t["bytes_per_launch"].items():
        assert name in bench.WORKLOADS or any(name in v for v in bench.WORKLOADS.values())
        assert nbytes > 10**9  # a 70B decode launch reads more than 1 GB


def test_percentiles(bench):
    assert bench._p10_p90([5, 1, 2, 3, 4, 6, 7, 8, 9, 10]) == [1, 9]
    assert bench._p10_p90([]) is None


def test_source_hash_ignores_comments_only(bench, tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_cache_270_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "pa_decode.cu").write_text("int a = 1;  // one\n\n// note\nint b = 2;\n")
    (csrc / "pa_device.cuh").write_text("#define X 3\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench._source_sha()
    (csrc / "pa_decode.cu").write_text("int a = 1;  // first\n// another note\nint b = 2;   \n")
    assert bench._source_sha() == h0
    (csrc / "pa_decode.cu").write_text("int a = 1;\nint b = 3;\n")
    assert bench._source_sha() != h0


def test_recorded_traffic_describes_the_current_decode_source(bench):
    """The DRAM traffic recorded from ncu is reported only while the decode
    kernel's code is the code it was taken on; a change to pa_decode.cu or
    pa_device.cuh (beyond comments) needs a new capture, or the line carries
    traffic null."""
    assert bench._source_sha() == bench.NCU_TRAFFIC["source_sha256"]
