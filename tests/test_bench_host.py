"""Host-side pieces of bench.py's JSON line, on CPU: the workload config both arms print, the
roofline object of the dominant kernel and the oracle's extrapolated full-step time."""
import json

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
    """The DRAM bytes per launch that the committed traffic file gives for the bench's three
    tensor-core kernels (full-size workload) lie within a few per cent of each kernel's
    compulsory traffic: every input read once, every output written once (a kernel that
    re-read K/V or Q/dO tiles from DRAM would show several times more)."""
    with open(bench.TRAFFIC_JSON) as f:
        got = {k: e["bytes_per_launch"] for k, e in json.load(f)["kernels"].items()}
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


def test_traffic_reader_takes_only_entries_of_the_current_sources(tmp_path):
    """profiled_traffic returns a kernel's bytes only while the recorded hash equals the hash
    of the kernel's current sources; a stale hash, a missing entry or a missing or malformed
    file gives None."""
    k = "fa_bwd_dq_tc_kernel<128>"
    cur = bench.kernel_source_sha256(k)
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"kernels": {k: {"bytes_per_launch": 1234, "source_sha256": cur}}}))
    assert bench.profiled_traffic(k, str(path)) == 1234
    path.write_text(json.dumps({"kernels": {k: {"bytes_per_launch": 1234,
                                                "source_sha256": "0" * 64}}}))
    assert bench.profiled_traffic(k, str(path)) is None
    assert bench.profiled_traffic("fa_fwd_tc_kernel<128>", str(path)) is None
    path.write_text("not json")
    assert bench.profiled_traffic(k, str(path)) is None
    assert bench.profiled_traffic(k, str(tmp_path / "absent.json")) is None


def test_source_hash_ignores_comments_but_not_code():
    """The hash that guards a traffic figure changes with the kernel's code only."""
    import re

    k = "fa_bwd_dq_tc_kernel<128>"
    h = bench.kernel_source_sha256(k)
    assert re.fullmatch(r"[0-9a-f]{64}", h)
    assert bench.kernel_source_sha256(k) == h


def test_fp8_entry_prefers_the_measured_gemm_and_keeps_the_assumed_ratio():
    peaks = {"bf16_tflops": 2000.0}
    e = bench.fp8_entry({"ms": 1.0, "tflops": 2400.0}, 3000.0, peaks)
    assert e["fp8_peak"] == 3000.0 and e["frac_of_fp8_peak"] == pytest.approx(0.8)
    assert e["fp8_peak_assumed"] == 4000.0 and e["frac_of_assumed_fp8_peak"] == pytest.approx(0.6)
    assert "measured" in e["fp8_peak_kind"]
    e = bench.fp8_entry({"ms": 1.0, "tflops": 2400.0}, None, peaks)
    assert e["fp8_peak"] == 4000.0 and e["frac_of_fp8_peak"] == pytest.approx(0.6)
    assert "assumed" in e["fp8_peak_kind"]
