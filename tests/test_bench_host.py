"""Host-side arithmetic of bench.py (no GPU): the roofline numerator and
denominator, and the rule that ties a DRAM-traffic capture to the kernel
sources it was taken on."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_of_the_bench_workload():
    # (M+N)*K operand bytes + (M+N)*K/32 scale bytes + M*N*2 BF16 output bytes
    assert bench.algorithmic_bytes(4096, 4096, 4096, "mxfp8", 2) == 68157440
    # MXFP4: half a byte per operand element; FP32 output
    assert bench.algorithmic_bytes(256, 256, 256, "mxfp4", 4) == 512 * 128 + 512 * 8 + 256 * 256 * 4


def test_mx_peaks_scale_the_measured_bf16_peak_by_the_nominal_ratio():
    assert bench.mx_peak_tflops("mxfp8", 1910.3) == pytest.approx(3820.6)
    assert bench.mx_peak_tflops("mxfp4", 1910.3) == pytest.approx(6 * 1910.3)


def _sources(tmp_path, texts):
    rels = []
    for i, t in enumerate(texts):
        (tmp_path / f"k{i}.cuh").write_text(t)
        rels.append(f"k{i}.cuh")
    return rels


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    code = "int f(int x) {\n  return x + 1;\n}\n"
    monkeypatch.setattr(bench, "KERNEL_SOURCES", _sources(tmp_path, [code]))
    h0 = bench.kernel_source_sha()
    commented = "// a note\nint f(int x) { /* inline\n note */\n  return x + 1;  // trailing\n}\n"
    monkeypatch.setattr(bench, "KERNEL_SOURCES", _sources(tmp_path, [commented]))
    assert bench.kernel_source_sha() == h0
    changed = "int f(int x) {\n  return x + 2;\n}\n"
    monkeypatch.setattr(bench, "KERNEL_SOURCES", _sources(tmp_path, [changed]))
    assert bench.kernel_source_sha() != h0


def test_traffic_is_read_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", _sources(tmp_path, ["int g();\n"]))
    f = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    entry = {"kernel_source_sha": bench.kernel_source_sha(), "dram_bytes_per_launch": 42.0e6, "note": "n"}
    f.write_text(json.dumps({"mxfp8_4096x4096x4096": entry}))
    assert bench.read_traffic("mxfp8", 4096, 4096, 4096) == (42.0e6, "n")
    assert bench.read_traffic("mxfp4", 4096, 4096, 4096) == (None, None)   # no capture of that case
    entry["kernel_source_sha"] = "0" * 16                                     # taken on other sources
    f.write_text(json.dumps({"mxfp8_4096x4096x4096": entry}))
    assert bench.read_traffic("mxfp8", 4096, 4096, 4096) == (None, None)

