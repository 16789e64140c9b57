"""e4m3 forward (fa_fwd_fp8) against the oracle on the values the codes stand for.

  * Integer scores with scale ln 2: every probability is a power of two (2^-8 .. 1), which
    e4m3 holds exactly, so the kernel's result is exact up to fp32 accumulation and the bf16
    rounding of O; checked at that tolerance.  This pins the whole data path (the S and P V
    products, the e4m3 P in Tensor Memory, the transposed V, the epilogue's descale).
  * Standard-normal inputs quantised per tensor: |O - O_ref| within the oracle's rounding
    bound (sum_j max(2^-4 P_ij, 2^-10 max P_i) |V_jc|, derived from e4m3's spacing) plus bf16
    rounding of O and an accumulation allowance; lse within 1e-3 (its scores are exact).
  * Full-size shapes (B=2 H=32 N=8192 and the bench's B=1 H=32 N=32000, causal) on sampled
    rows, and determinism.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import random_fp8

pytestmark = pytest.mark.gpu

LN2 = math.log(2.0)


def run(x, scale, causal):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward_fp8(q, k, v, x["q_descale"], x["k_descale"], x["v_descale"], scale=scale,
                            causal=causal)
    fa.fa_device_status()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def ref_of(x, scale, causal):
    return oracle.attention_fp8(x["q"], x["k"], x["v"], x["q_descale"], x["k_descale"],
                                x["v_descale"], scale, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 130), (2, 3, 257), (1, 1, 1000), (1, 1, 129)])
def test_integer_scores_are_exact(B, H, N, causal):
    x = random_fp8(B, H, N, 128, seed=N + B + causal, kind="integer")
    o, lse = run(x, LN2, causal)
    r = ref_of(x, LN2, causal)
    tol = 2.0 ** -8 * np.abs(r["o"]) + 1e-5 * r["pv_abs"] + 1e-6
    err = np.abs(o - r["o"])
    assert np.all(err <= tol), f"max err {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}"
    assert np.abs(lse - r["lse"]).max() <= 1e-4


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,in_scale", [(2, 2, 200, 1.0), (1, 4, 1000, 1.0), (1, 1, 700, 3.0),
                                            (1, 2, 385, 0.3)])
def test_random_inputs_within_the_rounding_bound(B, H, N, in_scale, causal):
    x = random_fp8(B, H, N, 128, seed=7 * N + causal, in_scale=in_scale)
    scale = 128 ** -0.5
    o, lse = run(x, scale, causal)
    r = ref_of(x, scale, causal)
    tol = r["bound"] + 2.0 ** -8 * (np.abs(r["o"]) + r["bound"]) + 1e-4 * r["pv_abs"] + 1e-6
    err = np.abs(o - r["o"])
    ratio = (err / tol).max()
    assert ratio <= 1.0, f"max err / tolerance {ratio:.3g}"
    assert np.abs(lse - r["lse"]).max() <= 1e-3


def test_uniform_weights_give_the_mean_of_v():
    x = random_fp8(1, 2, 300, 128, seed=3)
    x["q"] = torch.zeros_like(x["q"])
    for causal in (False, True):
        o, lse = run(x, 0.2, causal)
        v = oracle.e4m3_decode(oracle._codes(x["v"])) * x["v_descale"]
        for i in (0, 1, 128, 299):
            n = i + 1 if causal else 300
            mean = v[0, 1, :n].mean(axis=0)
            assert np.all(np.abs(o[0, 1, i] - mean) <= 2.0 ** -8 * np.abs(mean) + 1e-5)
            assert abs(lse[0, 1, i] - math.log(n)) <= 1e-4


def test_bench_shape_sampled_rows_and_determinism():
    B, H, N = 2, 32, 8192
    x = random_fp8(B, H, N, 128, seed=0, in_scale=0.5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    args = (q, k, v, x["q_descale"], x["k_descale"], x["v_descale"])
    o1, lse1 = fa.forward_fp8(*args, scale=128 ** -0.5, causal=True)
    o2, lse2 = fa.forward_fp8(*args, scale=128 ** -0.5, causal=True)
    fa.fa_device_status()
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
    rng = np.random.default_rng(0)
    rows = [(int(rng.integers(B)), int(rng.integers(H)), int(i))
            for i in list(rng.integers(0, N, 24)) + [0, 127, 128, N - 1]]
    r = oracle.attention_fp8_rows(x["q"], x["k"], x["v"], x["q_descale"], x["k_descale"],
                                  x["v_descale"], 128 ** -0.5, True, rows)
    o = o1.double().cpu().numpy()
    lse = lse1.double().cpu().numpy()
    for n, (b, h, i) in enumerate(rows):
        tol = (r["bound"][n] + 2.0 ** -8 * (np.abs(r["o"][n]) + r["bound"][n]) +
               1e-4 * r["pv_abs"][n] + 1e-6)
        assert np.all(np.abs(o[b, h, i] - r["o"][n]) <= tol), (b, h, i)
        assert abs(lse[b, h, i] - r["lse"][n]) <= 1e-3, (b, h, i)


def test_long_causal_sequence_sampled_rows():
    """The bench's shape (B=1, H=32, N=32000, causal: up to 250 key blocks per query tile),
    checked on sampled rows including the first and the last."""
    B, H, N = 1, 32, 32000
    x = random_fp8(B, H, N, 128, seed=5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward_fp8(q, k, v, x["q_descale"], x["k_descale"], x["v_descale"],
                            scale=128 ** -0.5, causal=True)
    fa.fa_device_status()
    rng = np.random.default_rng(1)
    rows = [(0, int(rng.integers(H)), int(i)) for i in list(rng.integers(0, N, 16)) + [0, N - 1]]
    r = oracle.attention_fp8_rows(x["q"], x["k"], x["v"], x["q_descale"], x["k_descale"],
                                  x["v_descale"], 128 ** -0.5, True, rows)
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    for n, (b, h, i) in enumerate(rows):
        tol = (r["bound"][n] + 2.0 ** -8 * (np.abs(r["o"][n]) + r["bound"][n]) +
               1e-4 * r["pv_abs"][n] + 1e-6)
        assert np.all(np.abs(o[b, h, i] - r["o"][n]) <= tol), (b, h, i)
        assert abs(lse[b, h, i] - r["lse"][n]) <= 1e-3, (b, h, i)


def test_fp8_argument_errors():
    x = random_fp8(1, 1, 64, 128, seed=1)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty((1, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as ei:
        fa.fa_fwd_fp8(q, k, v, o, None, 0.1, 1.0, 1.0, 1.0, False, small)
    assert ei.value.code == -4
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(1, 1, 64, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as ei:
        fa.fa_fwd_fp8(q, k, v, o, None, 0.1, math.inf, 1.0, 1.0, False, ws)
    assert ei.value.code == -1


def test_fp8_without_lse_gives_the_same_o():
    x = random_fp8(1, 2, 300, 128, seed=9)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    args = (x["q_descale"], x["k_descale"], x["v_descale"])
    o_ref, _ = fa.forward_fp8(q, k, v, *args, causal=True)
    o = torch.empty_like(o_ref)
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(1, 2, 300, 128), dtype=torch.uint8, device="cuda")
    fa.fa_fwd_fp8(q, k, v, o, None, 128 ** -0.5, *args, True, ws)
    fa.fa_device_status()
    assert torch.equal(o, o_ref)
