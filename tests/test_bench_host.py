"""The benchmark's host-side bookkeeping on CPU: the algorithmic bytes and
FLOPs each roofline divides by, the DRAM-traffic lookup that must go blank
once a kernel source changes, and the peak table's fallback."""

import json
import os

import bench


def test_algorithmic_bytes_per_launch():
    """Bytes a launch must move, against the per-launch figures of the
    workloads: read x once as bf16, write codes (E2M1: half a byte) plus one
    UE8M0 scale per 32 elements for each orientation."""
    assert bench.mx_quant_bytes(8192, 4096) == 67_108_864 + 2 * (33_554_432 + 1_048_576) == 136_314_880
    assert bench.mx_quant_bytes(8192, 4096, orient="row") == 67_108_864 + 33_554_432 + 1_048_576
    assert bench.mx_quant_bytes(4096, 14336, "e2m1", "row") == 117_440_512 + 29_360_128 + 1_835_008 == 148_635_648
    assert bench.pertensor_bytes(4096, 14336) == 234_881_024
    assert bench.pertensor_bytes(4096, 14336, "col") == 176_160_768


def test_gemm_flops():
    assert bench.gemm_flops(8192, 4096, 4096) == 274_877_906_944
    assert bench.gemm_flops(8192, 14336, 4096) == 962_072_674_304
    assert bench.gemm_flops(4096, 4096, 14336) == 481_036_337_152


def test_traffic_lookup_follows_the_kernel_source(tmp_path, monkeypatch):
    """A recorded DRAM count is reported only while the kernel file hashes
    to the value it was captured with, and only for its own workload."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({
        "k w": {"bytes_per_launch": 123, "source_sha": "abc"},
    }))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("k", "abc", "w") == 123
    assert bench.traffic_for("k", "abd", "w") is None
    assert bench.traffic_for("k", "abc", "other") is None
    os.remove(prof / "traffic.json")
    assert bench.traffic_for("k", "abc", "w") is None


def test_source_sha_changes_with_the_file(tmp_path, monkeypatch):
    csrc = tmp_path / "block_scaled_precision_02_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("a")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.source_sha("k.cu")
    (csrc / "k.cu").write_text("b")
    assert len(h1) == 16 and bench.source_sha("k.cu") != h1


def test_peaks_fall_back_when_not_measured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "of fallback" and peaks["hbm_gbs"] > 0 and peaks["bf16_tflops"] > 0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1.0, "bf16_tflops": 2.0}))
    peaks, src = bench.load_peaks()
    assert src == "of measured" and peaks["hbm_gbs"] == 1.0
