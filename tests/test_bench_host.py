"""Host logic of bench.py that needs no GPU: the nominal roofline of each
workload and the choice of the measured peak a kernel is judged against."""
from __future__ import annotations

import pytest

import bench
from warp_specialized_tma_gb300 import inputs

PEAKS = {"bf16_tflops": 1903.3, "bf16_tflops_sustained": 1712.9, "hbm_gbs": 6805.1}


@pytest.mark.parametrize("name,us,bound", [
    ("cube256", 0.049152, "hbm"),        # 2(3 * 256^2) bytes at 8 TB/s beats 2 * 256^3 FLOPs at 2.25 PF
    ("cube4096", 61.0839, "tensor"),
    ("cube8192", 488.6718, "tensor"),
    ("longk", 122.1679, "tensor"),
    ("ragged", 134.4357, "tensor"),
])
def test_nominal_roofline_of_the_workloads(name, us, bound):
    w = inputs.WORKLOADS[name]
    r = bench.nominal_roofline(w["M"], w["N"], w["K"])
    assert r["bound"] == bound
    assert r["us"] == pytest.approx(us, rel=1e-4)
    assert r["flops"] == 2.0 * w["M"] * w["N"] * w["K"]
    assert r["bytes"] == 2.0 * (w["M"] * w["K"] + w["N"] * w["K"] + w["M"] * w["N"])


def test_skinny_shapes_are_hbm_bound():
    for (m, n, k) in bench.SKINNY_SHAPES:
        assert bench.nominal_roofline(m, n, k)["bound"] == "hbm"


def test_peak_follows_the_length_of_the_timed_region():
    # a burst (the driver's 20 steps of cube8192 last ~11 ms) takes the burst peak
    burst = bench.measured_peak(PEAKS, "measured", "tensor", 0.011)
    assert burst["kind"] == "burst" and burst["peak"] == 1903.3 and burst["unit"] == "TFLOP/s"
    # seconds of back-to-back launches under the power cap take the sustained one
    sus = bench.measured_peak(PEAKS, "measured", "tensor", 3.5)
    assert sus["kind"] == "sustained" and sus["peak"] == 1712.9
    assert bench.measured_peak(PEAKS, "measured", "tensor", bench.SUSTAINED_MIN_S)["kind"] == "sustained"
    # an HBM-bound kernel is judged against the copy bandwidth, however long
    hbm = bench.measured_peak(PEAKS, "measured", "hbm", 0.011)
    assert hbm["kind"] == "hbm" and hbm["peak"] == 6805.1 and hbm["unit"] == "GB/s"


def test_fallback_peaks_when_the_measured_file_is_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback"
    assert peaks == bench.FALLBACK_PEAKS


def test_clock_summary_keeps_only_samples_inside_the_window():
    c = bench.NvmlClocks.__new__(bench.NvmlClocks)
    c.samples = [(0.5, 1000.0, 2070.0, 300.0, 0x0),
                 (1.1, 2070.0, 2070.0, 900.0, 0x0),
                 (1.2, 1980.0, 2070.0, 1300.0, 0x4),   # sw_power_cap
                 (1.3, 2010.0, 2070.0, 1200.0, 0x0),
                 (2.5, 900.0, 2070.0, 200.0, 0x8)]     # outside: hw_slowdown must not count
    s = c.summary(1.0, 2.0)
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2010.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert c.summary(3.0, 4.0)["samples"] == 0
