"""Host-side logic of bench.py, on the CPU: the FLOP convention, the input
checksums, and the lookup of recorded DRAM traffic, which must return a
figure only while the kernel's sources still hash as they did at capture."""

import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_flop_convention():
    # forward 4·B·H·S²·D/2, backward 2.5 × forward, step 3.5 × forward
    assert bench.fwd_flop(1, 32, 32768, 128) == 2.0 * 32 * 32768 ** 2 * 128
    assert abs(bench.fwd_flop(1, 32, 32768, 128) - 8.80e12) < 0.01e12
    assert bench.step_flop(2, 3, 100, 128) == 3.5 * bench.fwd_flop(2, 3, 100, 128)


def test_input_checksums_sum_the_first_2_20_elements():
    big = torch.ones((1 << 20) + 1000, dtype=torch.bfloat16).view(1, -1, 1, 1)
    small = torch.arange(10, dtype=torch.float32).to(torch.bfloat16)
    got = bench.input_checksums((("big", big), ("small", small)))
    assert got == {"big": float(1 << 20), "small": 45.0}


def test_recorded_traffic_needs_matching_source_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "long_context_causal_blockwise_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in (("attn_bwd.cu", "kernel v1\n"), ("common.cuh", "common\n"), ("tmem_ldst.cuh", "tmem\n")):
        (csrc / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash(bench.KERNEL_SOURCES["bwd_fused"])
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic_b1h32s32768.txt").write_text(
        "# comment lines and prose are skipped\n"
        f"bwd_fused {h} 2653056256\n"
        "dq_untile 0123456789abcdef 769436928\n")
    assert bench.recorded_traffic("bwd_fused") == 2653056256
    assert bench.recorded_traffic("dq_untile") is None  # recorded for other sources
    assert bench.recorded_traffic("attn_fwd") is None   # its sources are missing here
    (csrc / "attn_bwd.cu").write_text("kernel v2\n")
    assert bench.recorded_traffic("bwd_fused") is None  # the kernel changed since the capture


def test_tensor_peak_is_burst_unless_a_long_region_ran_power_capped():
    peaks = {"burst": 1904.1, "sustained": 1715.4, "hbm": 6743.6, "source": "measured"}
    # a sub-second region at full clocks: the burst figure
    assert bench.tensor_peak(peaks, 0.56, {"reasons": []}) == (1904.1, "burst")
    # the power cap alone in a short region does not change it, nor a long uncapped one
    assert bench.tensor_peak(peaks, 0.56, {"reasons": ["sw_power_cap"]}) == (1904.1, "burst")
    assert bench.tensor_peak(peaks, 20.0, {"reasons": []}) == (1904.1, "burst")
    # seconds under the power cap: the sustained figure, measured that way
    assert bench.tensor_peak(peaks, 20.0, {"reasons": ["sw_power_cap"]}) == (1715.4, "sustained")
    assert bench.tensor_peak(peaks, 20.0, None) == (1904.1, "burst")


def test_load_peaks_reads_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks()["source"] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        '{"hbm_gbs": 6743.6, "bf16_tflops": 1904.1, "bf16_tflops_sustained": 1715.4}')
    pk = bench.load_peaks()
    assert pk == {"burst": 1904.1, "sustained": 1715.4, "hbm": 6743.6, "source": "measured"}


def test_hbm_fields_divide_by_the_measured_copy_bandwidth():
    """The --rope and --ce lines: GB/s from algorithmic bytes and event ms, and
    the fraction of the measured HBM copy figure, with its source named."""
    peaks = {"burst": 1904.1, "sustained": 1715.4, "hbm": 6743.6, "source": "measured"}
    rec = bench.hbm_fields("fwd_", 8.59e9, 1.5, peaks)
    assert rec["fwd_gbs"] == pytest.approx(8.59e9 / 1.5e-3 / 1e9)
    assert rec["fwd_frac_of_hbm"] == pytest.approx(rec["fwd_gbs"] / 6743.6)
    assert rec["hbm_peak"] == 6743.6 and rec["hbm_peak_source"] == "measured"
    # every mode of bench.py reads the peaks through the dict load_peaks returns
    fb = bench.hbm_fields("", 1e9, 1.0, bench.load_peaks())
    assert fb["frac_of_hbm"] > 0 and isinstance(fb["hbm_peak"], float)
