"""Host-side helpers of bench.py: clock-sample parsing, the source-hash gate on committed DRAM
traffic, the peaks fallback and the audio duration a step delivers (no GPU needed)."""
from __future__ import annotations

import json
import os

import pytest

import bench
from dac_vocoder_decode_gb300 import workloads as W

FIELDS = bench.ClockSampler.FIELDS.split(",")


def smi_line(sm, smax, hw="Not Active", hw_th="Not Active", sw_th="Not Active", pcap="Not Active"):
    return ", ".join(["0", str(sm), str(smax), "812.45", "0x0000000000000004", hw, hw_th, sw_th, pcap])


def test_clock_summary_median_max_and_reasons():
    lines = [smi_line(1965, 2070), smi_line(1980, 2070, pcap="Active"), smi_line(1995, 2070),
             "", "index, clocks.sm [MHz]",  # stray header / blank lines are skipped
             smi_line("[N/A]", 2070), "0, 19"]  # unreadable clock, truncated last line
    out = bench.ClockSampler.summarize(lines)
    assert out["sm_mhz"] == 1980.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3


def test_clock_summary_reports_every_slowdown_reason():
    lines = [smi_line(1500, 2070, hw="Active"), smi_line(1400, 2070, hw_th="Active"),
             smi_line(1450, 2070, sw_th="Active")]
    out = bench.ClockSampler.summarize(lines)
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1450.0


def test_clock_summary_of_nothing():
    out = bench.ClockSampler.summarize([])
    assert out["sm_mhz"] is None and out["sm_max_mhz"] is None and out["samples"] == 0
    assert len(FIELDS) == 9  # the parser reads columns 1, 2 and 5..8 of exactly these fields


def make_tree(root, traffic_text):
    csrc = root / "dac_vocoder_decode_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("__global__ void k() {}\n")
    (root / "include").mkdir()
    (root / "include" / "k.h").write_text("void k(void);\n")
    (root / "profiles").mkdir()
    (root / "profiles" / "traffic_wl.md").write_text(traffic_text)


def test_measured_traffic_is_gated_by_the_source_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    make_tree(tmp_path, "")
    h = bench.source_hash()
    table = ("| layer | launches | ms | dram bytes | alg bytes |\n|---|---|---|---|---|\n"
             "| conv_in | 1 | 0.02 | 123456 | 100000 |\n| s0r0.conv1 | 1 | 0.15 | n/a | 5 |\n")
    (tmp_path / "profiles" / "traffic_wl.md").write_text(f"source hash: {h}\n\n{table}")
    assert bench.measured_traffic("wl", "conv_in")[0] == 123456
    assert bench.measured_traffic("wl", "s0r0.conv1") == (None, None)  # unparsable cell
    assert bench.measured_traffic("wl", "convT0") == (None, None)  # no such row
    assert bench.measured_traffic("other", "conv_in") == (None, None)  # no such summary
    # any change to a kernel source or the header retires the committed counters
    (tmp_path / "dac_vocoder_decode_gb300" / "csrc" / "k.cu").write_text("__global__ void k() {;}\n")
    assert bench.source_hash() != h
    assert bench.measured_traffic("wl", "conv_in") == (None, None)
    (tmp_path / "dac_vocoder_decode_gb300" / "csrc" / "k.cu").write_text("__global__ void k() {}\n")
    assert bench.measured_traffic("wl", "conv_in")[0] == 123456
    (tmp_path / "include" / "k2.h").write_text("\n")
    assert bench.measured_traffic("wl", "conv_in") == (None, None)


def test_long_decode_traffic_is_scaled_from_the_window_capture(tmp_path, monkeypatch):
    """music_long (15504 frames per item) takes music_window's (689 frames) per-launch DRAM
    bytes scaled by the frame ratio, and says so."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    make_tree(tmp_path, "")
    table = ("| layer | launches | ms | dram bytes | alg bytes |\n|---|---|---|---|---|\n"
             "| convT3 | 1 | 0.18 | 689000 | 1 |\n")
    (tmp_path / "profiles" / "traffic_music_window.md").write_text(
        f"source hash: {bench.source_hash()}\n\n{table}")
    value, src = bench.measured_traffic("music_long", "convT3")
    assert value == 15504000
    assert "music_window" in src and "15504/689" in src
    assert bench.measured_traffic("music_window", "convT3")[0] == 689000


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, kind = bench.load_peaks()
    assert kind == "fallback" and peaks["hbm_gbs"] == 6800.0 and peaks["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0}))
    peaks, kind = bench.load_peaks()
    assert kind == "measured" and peaks["hbm_gbs"] == 7000.0


def test_realtime_seconds_of_each_workload_kind():
    # stereo music window: one track of T * hop samples per pair of items
    wl = W.make_workload("music_window")
    assert wl.B == 2
    assert bench.realtime_seconds(wl, "music_window") == pytest.approx(wl.T * wl.arch.hop / 44100)
    # the small test decoders count every item as a track of its own
    wl = W.make_workload("tiny_cal")
    assert bench.realtime_seconds(wl, "tiny_cal") == pytest.approx(wl.B * wl.T * wl.arch.hop / 44100)
    # windowed batch: the stitched track, which covers the continuous latent it was cut from
    wl = W.make_workload("music_batch8")
    n_sides, _, frames = wl.continuous_latent.shape
    assert n_sides == 2
    assert bench.realtime_seconds(wl, "music_batch8") == pytest.approx(frames * wl.arch.hop / 44100)
    assert bench.realtime_seconds(wl, "music_batch8") < wl.B / 2 * wl.T * wl.arch.hop / 44100
    # speech items are mono tracks
    wl = W.make_workload("speech")
    assert bench.realtime_seconds(wl, "speech") == pytest.approx(wl.B * wl.T * wl.arch.hop / 24000)
    # encoder: stereo audio, one track per pair
    wl = bench.load_workload("encode_music_window", frames=4)
    B, _, L = wl.latent.shape
    assert bench.realtime_seconds(wl, "encode_music_window") == pytest.approx(B / 2 * L / 44100)


def test_cpu_threads_follows_omp(monkeypatch):
    monkeypatch.setenv("OMP_NUM_THREADS", "3")
    assert bench.cpu_threads() == 3
    monkeypatch.delenv("OMP_NUM_THREADS")
    assert bench.cpu_threads() == (os.cpu_count() or 1)


def test_clock_sampler_reads_a_fake_nvidia_smi(tmp_path, monkeypatch):
    """start()/stop() around a stand-in nvidia-smi on PATH that prints three samples and then
    keeps running until it is terminated, as the real one does with -lms."""
    fake = tmp_path / "nvidia-smi"
    rows = [smi_line(1900, 2070), smi_line(1920, 2070, pcap="Active"), smi_line(1940, 2070)]
    fake.write_text("#!/bin/sh\n" + "".join(f"echo '{r}'\n" for r in rows) + "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ.get('PATH', '')}")
    s = bench.ClockSampler(0)
    s.start()
    out = s.stop()
    assert out == {"sm_mhz": 1920.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # an empty directory: no nvidia-smi to start
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}


def test_tensor_peak_takes_the_sustained_figure_for_long_power_capped_runs():
    peaks = {"bf16_tflops": 1978.8, "bf16_tflops_sustained": 1739.1}
    assert bench.tensor_peak(peaks, 3.0, 4.2, ["sw_power_cap"]) == (1739.1 / 3.0, "sustained")
    # a short run, or one without the power cap, is held to the burst rate
    assert bench.tensor_peak(peaks, 3.0, 0.2, ["sw_power_cap"]) == (1978.8 / 3.0, "burst")
    assert bench.tensor_peak(peaks, 2.0, 4.2, []) == (1978.8 / 2.0, "burst")
    # without a measured sustained figure the fallback's
    assert bench.tensor_peak({}, 3.0, 4.2, ["sw_power_cap"])[0] == bench.FALLBACK_PEAKS["bf16_tflops_sustained"] / 3.0
