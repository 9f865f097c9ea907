"""Host logic of bench.py that needs no GPU: the roofline denominators, the
workload overrides.

MEASURED_PEAKS.json, written on each machine, holds the HBM copy GB/s and the
bf16 GEMM TFLOP/s (burst and sustained).  bench.py must use those numbers when
they are there, fall back to the stated figures when the file is absent, and
never fail the run because the file has another shape than expected.
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


def test_tensor_peak_is_burst_bf16_and_measured_or_nominal_fp8():
    import synth
    pk = {"hbm": 6500.0, "bf16": 1716.2, "bf16_sus": 1354.8, "source": "measured"}
    assert bench.tensor_peak(synth.get_config("v3"), pk)[0] == 1716.2
    assert bench.tensor_peak(synth.get_config("v3_fp8"), pk)[0] == 2 * 1716.2      # fp8 not measured
    pk["fp8"] = 3300.0
    assert bench.tensor_peak(synth.get_config("v3_fp8"), pk)[0] == 3300.0
    assert bench.tensor_peak(synth.get_config("v3"), pk)[0] == 1716.2


def test_roofline_fraction_recomputes_from_the_peak():
    """Both sides of the roofline recompute by hand from the algorithmic work,
    the stage time and the peaks; frac is the slower side's."""
    import numpy as np
    import synth
    cfg = synth.get_config("v3")
    pk = {"hbm": 6500.0, "bf16": 1716.2, "bf16_sus": 1354.8, "source": "measured"}
    counts = np.full(cfg.E, cfg.T * cfg.k // cfg.E, np.int32)
    r = bench.roofline(cfg, {"routed_gate_up": 4.0}, counts, pk)
    flops = 2 * cfg.T * cfg.k * cfg.d * 2 * cfg.inter
    nbytes = cfg.E * 2 * cfg.inter * cfg.d * 2 + cfg.T * cfg.k * (cfg.d + cfg.inter) * 2
    assert r["algorithmic_flops"] == flops and r["algorithmic_bytes"] == nbytes
    assert abs(r["tensor_frac"] - flops / 4e-3 / 1e12 / 1716.2) < 1e-4
    assert abs(r["hbm_frac"] - nbytes / 4e-3 / 1e9 / 6500.0) < 1e-4
    assert r["frac"] == max(r["tensor_frac"], r["hbm_frac"])
    assert r["bound"] == ("tensor" if r["tensor_frac"] >= r["hbm_frac"] else "hbm")
    assert abs(r["frac_of_sustained_bf16"] - flops / 4e-3 / 1e12 / 1354.8) < 1e-4


def test_both_arms_name_the_same_workload():
    import synth
    for name in ("v3", "v3_fp8", "mid"):
        cfg = synth.get_config(name)
        a, b = bench.workload_config(cfg), bench.workload_config(synth.get_config(name))
        assert a == b and a["workload"].startswith(("DeepSeek-V3-shaped", "mid-sized"))


def test_clock_sampler_without_a_gpu_id_reports_nothing():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc, s.uuid = None, None
    s.start()
    assert s.proc is None
    out = s.stop()
    assert out["sm_mhz"] is None and "not sampled" in out["reasons"][0]


def test_token_override_renames_the_workload():
    """--tokens T changes the batch and the name, so a DRAM-traffic figure
    recorded for the named size is never reported for another size."""
    import argparse
    a = argparse.Namespace(workload="v3", prec=None, tokens=2048)
    cfg = bench.layer_config(a)
    assert (cfg.T, cfg.name, cfg.d, cfg.E) == (2048, "v3_T2048", 7168, 256)
    assert bench.kernel_traffic("routed_gate_up", cfg.name) is None
    b = argparse.Namespace(workload="v3", prec="fp8", tokens=0)
    assert (bench.layer_config(b).T, bench.layer_config(b).prec, bench.layer_config(b).name) == (8192, "fp8", "v3")


def test_roofline_reports_both_hbm_denominators():
    """hbm_frac divides by the measured copy bandwidth, hbm_frac_of_nominal by
    the part's nominal 7.7 TB/s; both come from the same algorithmic bytes."""
    import numpy as np
    import synth
    cfg = synth.get_config("v3")
    counts = np.full(cfg.E, cfg.T * cfg.k // cfg.E)
    pk = dict(bench.FALLBACK_PEAKS, source="fallback")
    r = bench.roofline(cfg, {"routed_gate_up": 4.0}, counts, pk)
    B = bench.stage_work(cfg, counts)["routed_gate_up"][1]
    assert abs(r["hbm_frac"] - B / 4e-3 / 1e9 / pk["hbm"]) < 1e-4
    assert abs(r["hbm_frac_of_nominal"] - B / 4e-3 / 1e9 / bench.NOMINAL_HBM_GBS) < 1e-4
    assert r["hbm_frac_of_nominal"] < r["hbm_frac"]
