"""Host logic of the benchmark that needs no GPU: the recorded DRAM traffic
is only reported while the norm kernels' sources are the ones it was
captured from, and the CPU legs describe their host."""
import json
import os

import bench


def test_recorded_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    csrc = root / "rmsnorm_fp8_quantization_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (root / "profiles").mkdir()
    (csrc / "ring.cuh").write_text("// kernel\n")
    (csrc / "softmax.cu").write_text("// softmax\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    h = bench.kernel_source_hash()
    rec = {"norm_bwd": {"dram_bytes_per_launch": 123, "source_hash": h}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("norm_bwd") == 123
    assert bench.recorded_traffic("other_kernel") is None
    # the softmax translation unit is not part of the norm kernels
    (csrc / "softmax.cu").write_text("// softmax, changed\n")
    assert bench.kernel_source_hash() == h
    assert bench.recorded_traffic("norm_bwd") == 123
    # any change to the norm sources retires the record
    (csrc / "ring.cuh").write_text("// kernel, changed\n")
    assert bench.kernel_source_hash() != h
    assert bench.recorded_traffic("norm_bwd") is None


def test_host_description():
    d = bench.host_description()
    assert d["nproc"] == os.cpu_count() and d["cpu"] and d["arch"]
