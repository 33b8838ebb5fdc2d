"""Host-side logic of bench.py that needs no GPU: the clock-sample summary (median SM clock,
throttle reasons seen), the peaks file, the job throughput and the kernel-source key that
keeps a stored ncu traffic figure tied to the sources it was measured on."""

import json

import bench


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.lines = lines
    return s


def test_clock_summary_median_and_reasons():
    lines = [
        "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1390.2, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    out = _sampler(lines).summary()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3


def test_clock_summary_flags_thermal_slowdown_and_empty_input():
    lines = ["0, 1500, 2070, 1400, 0x40, Not Active, Active, Not Active, Not Active"]
    assert _sampler(lines).summary()["reasons"] == ["hw_thermal_slowdown"]
    empty = _sampler([]).summary()
    assert empty["sm_mhz"] is None and empty["samples"] == 0


def test_peaks_file_or_fallback(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6779.4,
                                                              "bf16_tflops": 1908.5}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._peaks() == (6779.4, 1908.5, "measured")
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    assert bench._peaks() == (6800.0, 1900.0, "fallback")


def test_job_value_counts_every_rank():
    assert bench.job_value(4096, 1, 0.5) == 4096 / 0.5e-3
    assert bench.job_value(4096, 4, 0.5) == 4 * 4096 / 0.5e-3


def test_kernel_key_tracks_the_gemm_sources():
    key = bench._kernel_key()
    parts = key.split(":")
    assert len(parts) == 2 and all(len(p) == 16 for p in parts)
    int(parts[0], 16), int(parts[1], 16)
