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
