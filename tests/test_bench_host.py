"""Host-side logic of bench.py (no GPU): the clock record and its rejection
rule, workload overrides, the JSON config both arms print, and the
whole-job arithmetic."""
import argparse
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

CAP, HW, THERM = (bench.ClockSampler.BITS[n]
                  for n in ("sw_power_cap", "hw_slowdown", "sw_thermal_slowdown"))


def _sampler(window=None):
    s = bench.ClockSampler(0)
    s.source = "test"
    s.window = window
    return s


def test_summary_keeps_only_the_timed_window():
    rows = [(0.5, 2032.0, 2032.0, 0), (1.0, 1300.0, 2032.0, CAP), (1.5, 1200.0, 2032.0, CAP),
            (2.0, 1400.0, 2032.0, CAP), (3.0, 2032.0, 2032.0, HW)]
    c = _sampler(window=(0.9, 2.1)).summary(rows)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 1300.0 and c["sm_min_mhz"] == 1200.0 and c["sm_max_mhz"] == 2032.0
    assert c["reasons"] == ["sw_power_cap"] and c["reason_samples"] == {"sw_power_cap": 3}


def test_summary_without_host_times_uses_every_row():
    rows = [(None, 1900.0, 2032.0, 0), (None, 1700.0, 2032.0, THERM)]
    c = _sampler(window=(5.0, 6.0)).summary(rows)
    assert c["samples"] == 2 and c["reasons"] == ["sw_thermal_slowdown"]


def test_summary_of_an_empty_window_is_unsampled():
    c = _sampler(window=(10.0, 11.0)).summary([(1.0, 2032.0, 2032.0, 0)])
    assert c["reasons"] == ["unsampled"] and c["sm_mhz"] is None


@pytest.mark.parametrize("clocks,rejected", [
    ({"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}, False),
    ({"sm_mhz": 1250.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"]}, False),
    ({"sm_mhz": 1900.0, "sm_max_mhz": 2032.0, "reasons": ["hw_slowdown"]}, True),
    ({"sm_mhz": 1900.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap", "hw_thermal_slowdown"]},
     True),
    ({"sm_mhz": 1900.0, "sm_max_mhz": 2032.0, "reasons": ["sw_thermal_slowdown"]}, True),
    # stuck well below the maximum with no reason at all: a leftover clock lock
    ({"sm_mhz": 1100.0, "sm_max_mhz": 2032.0, "reasons": []}, True),
    ({"sm_mhz": 1600.0, "sm_max_mhz": 2032.0, "reasons": []}, False),
    ({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}, False),
])
def test_clock_rejection_rule(clocks, rejected):
    assert bench.clocks_rejected(clocks) is rejected


def _args(**kw):
    a = dict(config="deepseek", tokens=0, experts=0, ffn_dim=0)
    a.update(kw)
    return argparse.Namespace(**a)


def test_workload_overrides():
    full = bench.resolve_cfg(_args())
    assert (full.T, full.N, full.f, full.fs) == (8192, 256, 2048, 2048)
    small = bench.resolve_cfg(_args(tokens=1024, experts=32))
    assert (small.T, small.N, small.d, small.f, small.k) == (1024, 32, 7168, 2048, 8)
    tiny_ffn = bench.resolve_cfg(_args(ffn_dim=64))
    assert (tiny_ffn.f, tiny_ffn.fs) == (64, 64)
    pre = bench.resolve_cfg(_args(config="mixtral_prefill", ffn_dim=64))
    assert (pre.f, pre.fs) == (64, 0)


def test_config_names_precision_and_options():
    cfg = bench.resolve_cfg(_args(config="capacity"))
    c = bench.config_dict(cfg, 1, fp8=True, fp8_down=True, reroute=2)
    assert c["fp8_gate_up"] and c["fp8_down"] and c["reroute_rounds"] == 2
    assert "re-routed in 2 rounds" in c["workload"] and "FP8 E4M3" in c["workload"]
    assert (c["T"], c["N"], c["capacity_factor"]) == (4096, 128, 1.25)
    assert bench.dtype_name(cfg, False, False) == "bf16"
    assert bench.dtype_name(cfg, True, False) == "e4m3 gate/up + bf16"
    assert bench.dtype_name(cfg, True, True) == "e4m3 experts + bf16"
    assert bench.dtype_name(bench.resolve_cfg(_args(config="tiny")), False, False) == "f32"
    plain = bench.config_dict(cfg, 4)
    assert plain["parallelism"] == "replicas x4 (no exchange)" and not plain["fp8_gate_up"]


def test_whole_job_value_counts_every_rank_over_the_slowest():
    assert bench.whole_job_value(1, 16384, 8.0) == pytest.approx(2.048e6)
    assert bench.whole_job_value(4, 16384, 8.0) == pytest.approx(8.192e6)
