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


def test_committed_traffic_matches_the_algorithmic_bytes():
    """The DRAM bytes per launch that the committed ncu summary gives for the bench's three
    tensor-core kernels (full-size workload) lie within a few per cent of each kernel's
    compulsory traffic: every input read once, every output written once (a kernel that
    re-read K/V or Q/dO tiles from DRAM would show several times more)."""
    import re

    text = open(bench.PROFILE_SUMMARY).read()
    got = {m.group(1): int(m.group(2))
           for m in re.finditer(r"traffic (\S+) bytes_per_launch=(\d+)", text)}
    assert set(got) == set(bench.KERNEL_SOURCES)
    B, H, N, d = 1, 32, 32000, 128
    t = B * H * N * d * 2          # one bf16 [B, H, N, d] tensor
    rows = B * H * N
    expect = {
        "fa_fwd_tc_kernel<128>": 3 * t + t + 4 * rows,           # Q, K, V -> O, LSE
        "fa_bwd_dkv_tc_kernel<128>": 4 * t + 8 * rows + 2 * t,   # Q, K, V, dO, LSE2, Delta -> dK, dV
        "fa_bwd_dq_tc_kernel<128>": 4 * t + 8 * rows + t,        # same inputs -> dQ
    }
    for k, bytes_ in got.items():
        assert 0.95 <= bytes_ / expect[k] <= 1.05, (k, bytes_, expect[k])
