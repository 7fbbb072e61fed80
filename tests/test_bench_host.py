"""Host-side pieces of bench.py that need no GPU: the roofline arithmetic of
the per-config entries, the clock poller's behaviour without NVML, and the
peak file reader."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


class _FakeRunner:
    peak_tf, peak_tf_sus, peak_bw = 2000.0, 1600.0, 8000.0


def test_roofline_tensor_bound():
    import bench
    # 1 TFLOP in 1 ms against a 2000 TFLOP/s burst and 1600 sustained peak; bytes far below HBM time
    r = bench.Runner.roofline(_FakeRunner(), 1.0, 1e12, 1e6)
    assert r["bound"] == "tensor"
    assert r["tflops"] == pytest.approx(1000.0)
    assert r["frac"] == pytest.approx(0.5)
    assert r["frac_sustained"] == pytest.approx(1000.0 / 1600.0)
    assert r["gbs"] == pytest.approx(1.0)


def test_roofline_hbm_bound_and_fp8_peak():
    import bench
    # 8 GB in 1 ms at 8000 GB/s is exactly the HBM roofline; FLOPs negligible
    r = bench.Runner.roofline(_FakeRunner(), 1.0, 1e9, 8e9)
    assert r["bound"] == "hbm"
    assert r["frac"] == pytest.approx(1.0) and r["frac_sustained"] == pytest.approx(1.0)
    # an FP8 kernel is measured against twice the bf16 peak
    r = bench.Runner.roofline(_FakeRunner(), 1.0, 2e12, 0, peak_mult=2.0)
    assert r["frac"] == pytest.approx(0.5)


def test_nvml_clocks_without_nvml_is_empty_not_an_error(monkeypatch):
    import ctypes
    import bench

    def no_lib(*a, **k):
        raise OSError("libnvidia-ml.so.1: not found")
    monkeypatch.setattr(ctypes, "CDLL", no_lib)
    c = bench.NvmlClocks(0).start()
    out = c.stop()
    assert out["sm_mhz"] is None and out["samples"] == 0


def test_measured_peaks_reads_the_driver_file(tmp_path, monkeypatch):
    import bench
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1883.2, "bf16_tflops_sustained": 1717.1,
                                                               "hbm_gbs": 6783.1}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (1883.2, 1717.1, 6783.1, "measured")
    os.remove(tmp_path / "MEASURED_PEAKS.json")
    tf, sus, bw, kind = bench.measured_peaks()
    assert kind == "fallback" and tf > sus > 0 and bw > 0
