"""Packed e4m3 forward (fa_fwd_fp8_varlen): variable-length sequences, grouped key/value heads,
the bottom-right causal mask and rows without keys, against the packed e4m3 oracle.

  * Integer scores with scale ln 2 (power-of-two weights, exact in e4m3): bf16 rounding
    tolerance only.
  * Standard-normal inputs: within the oracle's per-element rounding bound (as for the
    fixed-length e4m3 tests).
  * A packed batch of equal square sequences with Hkv = H gives the fixed-length call's
    results bit for bit (same tiles, same arithmetic, other addressing).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import random_fp8, random_fp8_varlen

pytestmark = pytest.mark.gpu

LN2 = math.log(2.0)

CASES = [
    # lens_q, lens_k, H, Hkv
    ([200], [200], 4, 4),
    ([1, 130, 0, 77], [300, 130, 50, 0], 4, 2),       # decode-like, square, no queries, no keys
    ([257, 5], [100, 600], 8, 1),                      # more queries than keys; MQA
    ([128, 129, 383], [256, 129, 1000], 6, 3),
]


def run(x, scale, causal):
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "cu_q", "cu_k")}
    o, lse = fa.forward_fp8_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"],
                                   x["max_q"], x["max_k"], x["q_descale"], x["k_descale"],
                                   x["v_descale"], scale=scale, causal=causal)
    fa.fa_device_status()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def ref_of(x, scale, causal):
    return oracle.attention_fp8_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"],
                                       x["q_descale"], x["k_descale"], x["v_descale"], scale,
                                       causal)


def check_lse(lse, ref, tol):
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref)), "rows without keys"
    fin = np.isfinite(ref)
    assert np.abs(lse[fin] - ref[fin]).max(initial=0.0) <= tol


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_packed_integer_scores_are_exact(case, causal):
    lens_q, lens_k, H, Hkv = CASES[case]
    x = random_fp8_varlen(lens_q, lens_k, H, Hkv, 128, seed=case + 10 * causal, kind="integer")
    o, lse = run(x, LN2, causal)
    r = ref_of(x, LN2, causal)
    tol = 2.0 ** -8 * np.abs(r["o"]) + 1e-5 * r["pv_abs"] + 1e-6
    err = np.abs(o - r["o"])
    assert np.all(err <= tol), f"max err {err.max():.3g}"
    check_lse(lse, r["lse"], 1e-4)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_packed_random_inputs_within_the_rounding_bound(case, causal):
    lens_q, lens_k, H, Hkv = CASES[case]
    x = random_fp8_varlen(lens_q, lens_k, H, Hkv, 128, seed=100 + case + 10 * causal)
    scale = 128 ** -0.5
    o, lse = run(x, scale, causal)
    r = ref_of(x, scale, causal)
    tol = r["bound"] + 2.0 ** -8 * (np.abs(r["o"]) + r["bound"]) + 1e-4 * r["pv_abs"] + 1e-6
    ratio = (np.abs(o - r["o"]) / tol).max()
    assert ratio <= 1.0, f"max err / tolerance {ratio:.3g}"
    check_lse(lse, r["lse"], 1e-3)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_square_batch_matches_fixed_length_bit_for_bit(causal):
    B, H, N = 3, 2, 300
    x = random_fp8(B, H, N, 128, seed=8)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    args = (x["q_descale"], x["k_descale"], x["v_descale"])
    o_f, lse_f = fa.forward_fp8(q, k, v, *args, causal=causal)
    pack = lambda t: t.permute(0, 2, 1, 3).reshape(B * N, H, 128).contiguous()  # noqa: E731
    cu = torch.arange(0, B * N + 1, N, dtype=torch.int32, device="cuda")
    o_p, lse_p = fa.forward_fp8_varlen(pack(q), pack(k), pack(v), cu, cu, N, N, *args,
                                       causal=causal)
    fa.fa_device_status()
    assert torch.equal(pack(o_f), o_p)
    assert torch.equal(lse_f.permute(1, 0, 2).reshape(H, B * N), lse_p)
