"""Host logic of bench.py that needs no GPU: the roofline denominators.

The driver writes MEASURED_PEAKS.json (HBM copy GB/s, bf16 GEMM TFLOP/s burst
and sustained).  bench.py must use those numbers when they are there, fall
back to the stated figures when the file is absent, and never fail the run
because the file has another shape than expected.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(tmp_path, obj):
    p = tmp_path / "MEASURED_PEAKS.json"
    p.write_text(json.dumps(obj) if not isinstance(obj, str) else obj)
    return str(p)


def test_absent_file_gives_the_fallback(tmp_path):
    pk = bench.peaks(str(tmp_path / "none.json"))
    assert pk["source"] == "fallback"
    assert (pk["hbm"], pk["bf16"], pk["bf16_sus"]) == (6400.0, 1800.0, 1400.0)


def test_plain_numbers_are_used(tmp_path):
    pk = bench.peaks(_write(tmp_path, {"hbm_gbs": 6464.0, "bf16_tflops": 1799.2, "bf16_tflops_sustained": 1390}))
    assert pk["source"] == "measured"
    assert (pk["hbm"], pk["bf16"], pk["bf16_sus"]) == (6464.0, 1799.2, 1390.0)


def test_nested_values_and_missing_sustained(tmp_path):
    pk = bench.peaks(_write(tmp_path, {"hbm_gbs": {"value": 6500, "unit": "GB/s"},
                                       "bf16_tflops": {"median": "1800.5"}}))
    assert pk["source"] == "measured"
    assert (pk["hbm"], pk["bf16"], pk["bf16_sus"]) == (6500.0, 1800.5, 1800.5)


def test_unreadable_file_falls_back_and_says_so(tmp_path):
    for bad in ("{not json", {"hbm": 1}, {"hbm_gbs": None, "bf16_tflops": 1}, {"hbm_gbs": {"x": 1}, "bf16_tflops": 2}):
        pk = bench.peaks(_write(tmp_path, bad))
        assert pk["source"].startswith("fallback (MEASURED_PEAKS.json unreadable")
        assert pk["hbm"] == 6400.0
