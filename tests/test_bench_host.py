"""Host-side pieces of bench.py's JSON line, on CPU: the workload config both arms print, the
roofline object of the dominant kernel and the oracle's extrapolated full-step time."""
import pytest

import bench
from exact_attention_25_gb300 import perfmodel
from exact_attention_25_gb300.inputs import WORKLOADS


def test_both_arms_name_the_same_workload():
    w = WORKLOADS[bench.WORKLOAD]
    cfg = bench.workload_config(w, 1)
    assert (cfg["B"], cfg["H"], cfg["N"], cfg["d"], cfg["causal"]) == (1, 32, 32000, 128, True)
    assert cfg["scale"] == pytest.approx(128 ** -0.5)
    assert cfg["parallelism"] == "single GPU"
    assert bench.workload_config(w, 4)["parallelism"] == "replicas4"
    assert "model" not in cfg


def test_roofline_fractions_against_burst_and_sustained_peaks():
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    r = bench.roofline_entry("k", 1200.0, peaks, "measured", 123)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["peak"] == 2000.0 and r["frac"] == pytest.approx(0.6)
    assert r["peak_sustained"] == 1600.0 and r["frac_sustained"] == pytest.approx(0.75)
    assert r["traffic"] == 123
    r = bench.roofline_entry("k", 950.0, {"bf16_tflops": 1900.0}, "fallback", None)
    assert r["frac"] == pytest.approx(0.5) and "frac_sustained" not in r
    assert r["traffic"] is None and "fallback" in r["peak_kind"]


def test_oracle_extrapolation_scales_with_the_workload_flops():
    w = WORKLOADS[bench.WORKLOAD]
    flops = perfmodel.fwd_flops(1, 32, 32000, 128, True) * 3.5  # forward + 2.5 x forward
    assert bench.oracle_full_step_seconds(w, 1.0) == pytest.approx(flops / 1e12)
    assert bench.oracle_full_step_seconds(w, 2.0) == pytest.approx(flops / 2e12)
