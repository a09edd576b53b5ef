"""bench.py's roofline denominators: read from the measured peaks file in any
of the shapes it may take, or the fallback figures when it is absent or
unusable.  CPU only."""
import json

import bench


def write(tmp_path, obj):
    p = tmp_path / "peaks.json"
    p.write_text(obj if isinstance(obj, str) else json.dumps(obj))
    return str(p)


def test_flat_file(tmp_path):
    peaks, src = bench.load_peaks(write(tmp_path, {"hbm_gbs": 6782.0, "bf16_tflops": 1887.0,
                                                   "bf16_tflops_sustained": 1705.0}))
    assert src == "measured"
    assert peaks == {"hbm_gbs": 6782.0, "bf16_tflops": 1887.0, "bf16_tflops_sustained": 1705.0}


def test_nested_file_and_missing_sustained(tmp_path):
    peaks, src = bench.load_peaks(write(tmp_path, {"gpu": "GB300", "peaks": {"hbm_gbs": 6500, "bf16_tflops": 1800}}))
    assert src == "measured"
    assert peaks["hbm_gbs"] == 6500.0 and peaks["bf16_tflops"] == 1800.0
    assert peaks["bf16_tflops_sustained"] == 1800.0  # burst stands in when no sustained figure is given


def test_incomplete_or_broken_file_falls_back(tmp_path):
    for obj in ({"hbm_gbs": 6500}, "{not json", []):
        peaks, src = bench.load_peaks(write(tmp_path, obj))
        assert src == "fallback" and peaks == bench.FALLBACK_PEAKS


def test_absent_file_falls_back(tmp_path):
    peaks, src = bench.load_peaks(str(tmp_path / "none.json"))
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS


def _traffic_file(tmp_path, fingerprint, traffic="1625250000"):
    p = tmp_path / "traffic.txt"
    p.write_text("attn traffic summary\n"
                 "  indented: lines are ignored\n"
                 f"traffic_bytes_per_launch_480p_group28: {traffic}\n"
                 f"attention_sources_sha256_16: {fingerprint}\n")
    return str(p)


def test_traffic_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    """The committed DRAM capture is reported only while the attention sources
    still have the fingerprint recorded with it; otherwise traffic is null."""
    fp = bench.attention_fingerprint()
    assert len(fp) == 16 and int(fp, 16) >= 0
    monkeypatch.setattr(bench, "TRAFFIC_FILE", _traffic_file(tmp_path, fp))
    traffic, src = bench.read_traffic()
    assert traffic == 1625250000.0 and "same kernel sources" in src
    monkeypatch.setattr(bench, "TRAFFIC_FILE", _traffic_file(tmp_path, "0" * 16))
    traffic, src = bench.read_traffic()
    assert traffic is None and "other attention sources" in src
    monkeypatch.setattr(bench, "TRAFFIC_FILE", _traffic_file(tmp_path, fp, traffic="n/a"))
    assert bench.read_traffic() == (None, None)
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.txt"))
    assert bench.read_traffic() == (None, None)


def test_committed_traffic_capture_matches_the_current_sources():
    """The committed capture was taken on the attention sources as they are:
    if the kernel changes, the capture has to be taken again."""
    traffic, src = bench.read_traffic()
    assert traffic is not None and traffic > 4 * 51200 * 28 * 128 * 2, src


def test_clock_summary_of_an_nvidia_smi_capture():
    """Median clock and power, and every throttle reason that was active in
    any sample; rows that do not parse are skipped."""
    hdr = ("index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw.instant [W], clocks_event_reasons.active, "
           "clocks_event_reasons.hw_slowdown, clocks_event_reasons.hw_thermal_slowdown, "
           "clocks_event_reasons.sw_thermal_slowdown, clocks_event_reasons.sw_power_cap")
    rows = ["0, 1897 MHz, 2070 MHz, 1240.50 W, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1905 MHz, 2070 MHz, 1251.00 W, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1850 MHz, 2070 MHz, 1238.25 W, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, [N/A], 2070 MHz, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",
            "truncated, row"]
    out = bench.ClockSampler.summarize("\n".join([hdr] + rows) + "\n")
    assert out == {"sm_mhz": 1897.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                   "power_w": 1240.5}
    assert bench.ClockSampler.summarize(hdr + "\n") is None
    assert bench.ClockSampler.summarize("") is None
