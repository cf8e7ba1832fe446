"""The bench line's `roofline.traffic` comes from a recorded ncu capture that counts only while
the kernel's sources are unchanged.  These tests run on the CPU against a fake source tree."""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture()
def bench(tmp_path, monkeypatch):
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    csrc = tmp_path / "exact_flow_recurrence_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text('#include "a.cuh"\n#include <cuda.h>\n__global__ void k_x() {}\n')
    (csrc / "a.cuh").write_text('#pragma once\n  #include "b.cuh"\nint a;\n')
    (csrc / "b.cuh").write_text("#pragma once\nint b;\n")
    (csrc / "other.cuh").write_text("int unrelated;\n")
    monkeypatch.setattr(mod, "ROOT", str(tmp_path))
    monkeypatch.setattr(mod, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    return mod, csrc


def _csv(path, rows):
    lines = ['"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"']
    for i, name, metric, value in rows:
        lines.append(f'"{i}","{name}","{metric}","byte","{value}"')
    path.write_text("==PROF== noise before the table\n" + "\n".join(lines) + "\n")


def test_hash_covers_included_headers_only(bench):
    mod, csrc = bench
    h0 = mod._source_sha1("k.cu")
    assert h0 == mod._source_sha1("k.cu")
    (csrc / "other.cuh").write_text("int unrelated = 1;\n")   # not included: no change
    assert mod._source_sha1("k.cu") == h0
    (csrc / "b.cuh").write_text("#pragma once\nint b = 2;\n")   # included through a.cuh
    assert mod._source_sha1("k.cu") != h0


def test_record_then_invalidate(bench, tmp_path):
    mod, csrc = bench
    _csv(tmp_path / "cap.csv", [
        ("0", "at::fill", "dram__bytes_read.sum", "999"),
        ("1", "k_x<0>", "dram__bytes_read.sum", "1,000"),
        ("1", "k_x<0>", "dram__bytes_write.sum", "500"),
        ("2", "k_x<0>", "dram__bytes_read.sum", "1200"),
        ("2", "k_x<0>", "dram__bytes_write.sum", "300"),
        ("2", "k_x<0>", "gpu__time_duration.sum", "7"),
    ])
    mod.record_traffic(str(tmp_path / "cap.csv"), "k_x@w", "k_x", "k.cu", "ncu ...")
    ent = json.loads((tmp_path / "traffic.json").read_text())["entries"]["k_x@w"]
    assert ent["launches_captured"] == 2 and ent["dram_bytes_per_launch"] == 1500
    assert mod.measured_traffic("k_x@w") == 1500
    assert mod.measured_traffic("missing@w") is None
    (csrc / "a.cuh").write_text('#pragma once\n#include "b.cuh"\nint a = 3;\n')
    assert mod.measured_traffic("k_x@w") is None


def test_roofline_times_the_dominant_kernel_when_it_carries_the_call(bench):
    mod, _ = bench
    fused = {"efla_zero_flags": {"ms": 0.005, "per_call": 1.0}, "efla_tc_fused": {"ms": 0.074, "per_call": 1.0}}
    dom, t, path = mod.roofline_timing(fused)
    assert dom == "efla_tc_fused" and t == pytest.approx(0.074) and path == pytest.approx(0.079)
    two = {"efla_tc_tmat": {"ms": 0.04, "per_call": 1.0}, "efla_tc_fwd": {"ms": 0.068, "per_call": 1.0}}
    dom, t, path = mod.roofline_timing(two)   # no kernel carries 90%: the whole call
    assert dom == "efla_tc_fwd" and t == pytest.approx(0.108) and path == pytest.approx(0.108)
    one = {"efla_decode_step": {"ms": 0.08, "per_call": 2.0}}
    assert mod.roofline_timing(one) == ("efla_decode_step", pytest.approx(0.16), pytest.approx(0.16))
