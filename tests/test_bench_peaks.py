"""The bench's roofline denominators: measured figures from MEASURED_PEAKS.json
key by key, the fallback figures for anything missing or malformed."""

import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_no_file_gives_fallback(tmp_path):
    pk, src = bench.peaks(str(tmp_path))
    assert src == "fallback" and pk == bench.FALLBACK


def test_measured_keys_override_one_by_one(tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1850.5, "other": 1}))
    pk, src = bench.peaks(str(tmp_path))
    assert src == "measured" and pk["bf16_tflops"] == 1850.5
    assert pk["hbm_gbs"] == bench.FALLBACK["hbm_gbs"]
    assert pk["bf16_tflops_sustained"] == bench.FALLBACK["bf16_tflops_sustained"]


def test_records_and_malformed_values(tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"bf16_tflops": {"value": 1790.0}, "hbm_gbs": "n/a", "bf16_tflops_sustained": -3}))
    pk, src = bench.peaks(str(tmp_path))
    assert src == "measured" and pk["bf16_tflops"] == 1790.0
    assert pk["hbm_gbs"] == bench.FALLBACK["hbm_gbs"]
    assert pk["bf16_tflops_sustained"] == bench.FALLBACK["bf16_tflops_sustained"]


def test_unreadable_file_gives_fallback(tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    pk, src = bench.peaks(str(tmp_path))
    assert src == "fallback" and pk == bench.FALLBACK
