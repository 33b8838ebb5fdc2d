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
    tag, a, b = key.split(":")
    assert tag == "code" and len(a) == 16 and len(b) == 16
    int(a, 16), int(b, 16)


def test_kernel_key_ignores_comments_but_not_code():
    src = "int f(int x) {\n  // a note\n  return x + 1;  /* another\n note */\n}\n"
    same = "int f(int x) {\n  // the note, reworded\n  return x + 1;\n}\n"
    other = "int f(int x) {\n  // a note\n  return x + 2;\n}\n"
    assert bench._strip_comments(src) == bench._strip_comments(same)
    assert bench._strip_comments(src) != bench._strip_comments(other)


class _Inp:
    def __init__(self, T, H, E, I, k):
        self.T, self.H, self.E, self.I, self.k = T, H, E, I, k


def test_stage_bytes_count_each_tensor_once():
    inp = _Inp(4096, 2048, 64, 768, 8)
    b = bench.stage_bytes(inp)
    r = 4096 * 8
    assert b["combine"] == r * 2048 * 2 + r * 8 + 4096 * 2048 * 2
    assert b["quant_g128"] == 4096 * 2048 * 3 + 4096 * 16 * 4
    assert b["topk_gate"] == 4096 * 64 * 4 + r * 8
    # the fused routing stage reads bf16 once instead of the codes, so it moves T*H bytes more
    # than the separate permute minus the separate quantization's own output
    assert b["permute_quant"] - b["permute"] == 4096 * 2048 - 4096 * 16 * 4


def test_layer_work_counts_only_experts_with_rows():
    inp = _Inp(64, 256, 8, 512, 2)
    f_all, b_all = bench.layer_work(inp, [16] * 8)
    f_half, b_half = bench.layer_work(inp, [32, 0] * 4)
    assert f_all == f_half == 2.0 * 128 * (1024 * 256 + 256 * 512)
    bank = 1024 * 256 // 2 + 256 * 512 // 2 + (1024 * 2 + 256 * 4) * 4
    assert b_all - b_half == 4 * bank


def test_roofline_fraction_takes_the_slower_floor():
    # 1 TFLOP at 1000 TF/s = 1 ms; 1 GB at 1000 GB/s = 1 ms; measured 2 ms -> 0.5
    frac, bound = bench.roofline_frac(1e12, 1e9, 2.0, 1000.0, 1000.0)
    assert abs(frac - 0.5) < 1e-12
    frac, bound = bench.roofline_frac(1e12, 4e9, 8.0, 1000.0, 1000.0)
    assert abs(frac - 0.5) < 1e-12 and bound == "hbm"
    frac, bound = bench.roofline_frac(4e12, 1e9, 8.0, 1000.0, 1000.0)
    assert abs(frac - 0.5) < 1e-12 and bound == "tensor"


def test_cpu_info_reports_the_core_count():
    import os
    info = bench.cpu_info()
    assert info["nproc"] == os.cpu_count() and info["machine"]


def test_stage_write_bytes_within_totals():
    inp = _Inp(16384, 4096, 128, 1536, 8)
    tot, wr = bench.stage_bytes(inp), bench.stage_write_bytes(inp)
    assert set(tot) == set(wr)
    for name in tot:
        assert 0 < wr[name] < tot[name], name
    # the permuted copies write k rows per token read
    assert wr["permute_quant"] > 4 * (tot["permute_quant"] - wr["permute_quant"])


def test_memory_floor_takes_the_slower_bound():
    # 1 GB read + 1 GB written: copy-bound at 2 GB / 6000 GB/s
    assert bench.memory_floor_ms(2e9, 1e9, 6000.0, 4000.0) == 2e9 / 6000.0 / 1e6
    # 0.2 GB read + 1.8 GB written: write-bound at 1.8 GB / 4000 GB/s
    assert bench.memory_floor_ms(2e9, 1.8e9, 6000.0, 4000.0) == 1.8e9 / 4000.0 / 1e6
