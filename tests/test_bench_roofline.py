"""Host-side roofline arithmetic of bench.py: which measured peak divides the achieved rate, the
fractions reported beside it, the spec peak from the measured tensor-core rate, and the traffic
record that goes stale with the kernel source."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "measured"}


def test_tensor_roofline_burst_and_sustained():
    burst = bench.tensor_roofline(950.0, PEAKS, "k", None)
    assert burst["peak"] == 1900.0 and burst["frac"] == pytest.approx(0.5)
    assert burst["frac_of_sustained_peak"] == pytest.approx(950.0 / 1700.0, abs=1e-4)
    sus = bench.tensor_roofline(850.0, PEAKS, "k", 123.0, sustained=True)
    assert sus["peak"] == 1700.0 and sus["frac"] == pytest.approx(0.5)
    assert sus["frac_of_burst_peak"] == pytest.approx(850.0 / 1900.0, abs=1e-4)
    assert sus["traffic"] == 123.0 and "sustained" in sus["peak_source"]


def test_tensor_roofline_fp8_doubles_both_peaks():
    r = bench.tensor_roofline(1900.0, PEAKS, "k", None, fp8=True, sustained=True)
    assert r["peak"] == 3400.0 and r["frac"] == pytest.approx(1900.0 / 3400.0, abs=1e-4)
    assert r["frac_of_burst_peak"] == pytest.approx(0.5)
    assert "x 2" in r["peak_source"]


def test_hbm_roofline():
    r = bench.hbm_roofline(3400.0, PEAKS, "k", None)
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(0.5) and r["frac_of_8TBps"] == pytest.approx(0.425)


def test_spec_peak_from_the_measured_rate():
    sp = bench.SpecPeak.__new__(bench.SpecPeak)
    sp.n_sm, sp.rate, sp.lo, sp.hi, sp.max_mhz, sp.sampled_mhz = 152, 8192.0, 8190.0, 8194.0, 2000.0, 1000.0
    assert sp.tflops(2000.0) == pytest.approx(152 * 8192.0 * 2000e6 / 1e12)
    rec = sp.record(sp.tflops(1000.0))
    assert rec["frac_of_spec_at_sampled_clock"] == pytest.approx(1.0)
    assert rec["frac_of_spec_at_max_clock"] == pytest.approx(0.5)
    assert rec["achieved_flop_per_sm_cycle"] == pytest.approx(8192.0, abs=0.1)


def test_traffic_record_goes_stale_with_the_source(tmp_path, monkeypatch):
    csrc = tmp_path / "attention_attn_fwd_03_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("kernel v1")
    import hashlib
    sha = hashlib.sha256(b"kernel v1").hexdigest()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"key": {"dram_bytes_per_launch": 42.0, "source_sha256": sha}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("k.cu", "key") == 42.0
    assert bench.traffic_record("k.cu", "other") is None
    (csrc / "k.cu").write_text("kernel v2")
    assert bench.traffic_record("k.cu", "key") is None
