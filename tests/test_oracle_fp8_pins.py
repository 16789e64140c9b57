"""Pins of the oracle's e4m3 part (CPU): the code table against the format's closed forms and
torch's float8_e4m3fn conversion, the descale factors against invariances of the definition,
and the rounding bound against a step-by-step simulation of online softmax with e4m3
probabilities, which the bound must cover and which a bound without its subnormal term
must fail."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_25_gb300.inputs import random_fp8


def test_e4m3_code_table_closed_forms():
    v = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x00] == 0.0 and math.copysign(1.0, v[0x80]) == -1.0
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9   # subnormals m/8 * 2^-6
    assert v[0x08] == 2.0 ** -6                                 # smallest normal
    assert v[0x38] == 1.0 and v[0xB8] == -1.0 and v[0x40] == 2.0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0              # largest finite
    assert math.isnan(v[0x7F]) and math.isnan(v[0xFF])
    assert np.isfinite(v).sum() == 254
    # the finite positive values are strictly increasing in code order
    pos = v[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)


def test_e4m3_code_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_decode(codes.numpy()), ref, equal_nan=True)


def test_uniform_probabilities_give_closed_forms():
    """Q = 0: every visible key weighs the same, so O_i is the mean of the visible V rows and
    lse_i = ln(count) (the closed form of the bf16 pins, through the e4m3 decoding)."""
    x = random_fp8(1, 2, 37, 128, seed=1)
    q8 = torch.zeros_like(x["q"])
    v = oracle.e4m3_decode(oracle._codes(x["v"])) * x["v_descale"]
    for causal in (False, True):
        r = oracle.attention_fp8(q8, x["k"], x["v"], 1.0, x["k_descale"], x["v_descale"], 0.3,
                                 causal)
        for i in (0, 5, 36):
            n = i + 1 if causal else 37
            assert np.allclose(r["o"][0, 1, i], v[0, 1, :n].mean(axis=0), rtol=1e-12, atol=1e-12)
            assert abs(r["lse"][0, 1, i] - math.log(n)) < 1e-12


def test_descale_factors_compose_like_the_definition():
    """Only the products scale * q_descale * k_descale and v_descale matter; O and the bound are
    linear in v_descale."""
    x = random_fp8(1, 1, 64, 128, seed=2)
    a = oracle.attention_fp8(x["q"], x["k"], x["v"], 2.0, 3.0, 1.0, 0.01, True)
    b = oracle.attention_fp8(x["q"], x["k"], x["v"], 1.0, 1.0, 1.0, 0.06, True)
    c = oracle.attention_fp8(x["q"], x["k"], x["v"], 6.0, 1.0, 2.5, 0.01, True)
    assert np.allclose(a["o"], b["o"], rtol=1e-12, atol=1e-14)
    assert np.allclose(a["lse"], b["lse"], rtol=1e-12, atol=1e-12)
    assert np.allclose(c["o"], 2.5 * a["o"], rtol=1e-12, atol=1e-14)
    assert np.allclose(c["bound"], 2.5 * a["bound"], rtol=1e-12, atol=1e-14)
    rows = oracle.attention_fp8_rows(x["q"], x["k"], x["v"], 2.0, 3.0, 1.0, 0.01, True,
                                     [(0, 0, 0), (0, 0, 17), (0, 0, 63)])
    for n, (_, _, i) in enumerate([(0, 0, 0), (0, 0, 17), (0, 0, 63)]):
        assert np.allclose(rows["o"][n], a["o"][0, 0, i], rtol=1e-12, atol=1e-14)
        assert abs(rows["lse"][n] - a["lse"][0, 0, i]) < 1e-12
        assert np.allclose(rows["bound"][n], a["bound"][0, 0, i], rtol=1e-12, atol=1e-14)


def simulate_online_e4m3(x, v, block=128, threshold=8.0):
    """One row: online softmax over key blocks in log2 units x (scores * scale * log2 e), the
    reference maximum moved only when a block's maximum exceeds it by more than `threshold`,
    probabilities rounded to e4m3 (torch, nearest even) before they weigh V, O divided by the
    sum of the unrounded probabilities."""
    m, l = -math.inf, 0.0
    acc = np.zeros(v.shape[1])
    for j0 in range(0, len(x), block):
        xb, vb = x[j0:j0 + block], v[j0:j0 + block]
        mt = xb.max()
        if mt > m + threshold:
            alpha = 0.0 if m == -math.inf else 2.0 ** (m - mt)
            m, l, acc = mt, l * alpha, acc * alpha
        p = np.exp2(xb - m)
        l += p.sum()
        pq = torch.from_numpy(p).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        acc = acc + pq @ vb
    return acc / l


@pytest.mark.parametrize("seed", range(6))
def test_rounding_bound_covers_simulated_online_softmax(seed):
    rng = np.random.default_rng(seed)
    N, d = 700, 16
    x = rng.normal(size=N) * [1.0, 4.0, 12.0, 0.3, 25.0, 6.0][seed]
    if seed == 5:
        x = np.sort(x)  # increasing scores: the reference maximum moves often
    v = rng.normal(size=(N, d))
    P = np.exp2(x - x.max())
    P /= P.sum()
    o = P @ v
    bound = np.maximum(P / 16.0, P.max() / 1024.0) @ np.abs(v)
    err = np.abs(simulate_online_e4m3(x, v) - o)
    assert np.all(err <= bound * (1 + 1e-9) + 1e-15), (err / bound).max()


def test_bound_needs_its_subnormal_term():
    """Many small weights near the subnormal range: their rounding error adds up beyond
    2^-4 P, so a bound without the 2^-10 term fails while the full bound holds."""
    N = 1024
    x = np.full(N, -10.0 + math.log2(1.4))   # p ~ 1.4 * 2^-10, rounds to 2^-9
    x[0] = 0.0
    v = np.ones((N, 1))
    v[0] = 0.0
    P = np.exp2(x)
    P /= P.sum()
    o = P @ v
    err = np.abs(simulate_online_e4m3(x, v) - o)
    full = np.maximum(P / 16.0, P.max() / 1024.0) @ np.abs(v)
    assert np.all(err <= full)
    assert np.any(err > (P / 16.0) @ np.abs(v))


def _dec(t, s):
    return oracle.e4m3_decode(oracle._codes(t)) * s


@pytest.mark.parametrize("causal", [False, True])
def test_packed_e4m3_oracle_matches_the_c_oracle(causal):
    """The packed e4m3 oracle (numpy, per sequence and head) against the C oracle's
    attention_varlen on the decoded values: two implementations of the same definition,
    including grouped heads, Nq != Nk in both directions and empty sequences."""
    from exact_attention_25_gb300.inputs import random_fp8_varlen

    x = random_fp8_varlen([3, 0, 40, 7, 12], [5, 9, 30, 0, 12], 4, 2, 128, seed=1)
    r = oracle.attention_fp8_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"],
                                    x["q_descale"], x["k_descale"], x["v_descale"], 0.09, causal)
    ref = oracle.attention_varlen(_dec(x["q"], x["q_descale"]), _dec(x["k"], x["k_descale"]),
                                  _dec(x["v"], x["v_descale"]), x["cu_q"], x["cu_k"], 0.09, causal)
    assert np.allclose(r["o"], ref["o"], rtol=0, atol=1e-12)
    assert np.array_equal(np.isneginf(r["lse"]), np.isneginf(ref["lse"]))
    fin = np.isfinite(ref["lse"])
    assert np.allclose(r["lse"][fin], ref["lse"][fin], rtol=0, atol=1e-12)


def test_packed_e4m3_oracle_reduces_to_the_fixed_one():
    """One square sequence with as many key/value heads as query heads is the fixed-length
    problem: o, lse, bound and pv_abs agree with attention_fp8."""
    from exact_attention_25_gb300.inputs import random_fp8_varlen

    x = random_fp8_varlen([50], [50], 3, 3, 128, seed=2)
    r = oracle.attention_fp8_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"],
                                    x["q_descale"], x["k_descale"], x["v_descale"], 0.1, True)
    f = oracle.attention_fp8(x["q"].permute(1, 0, 2)[None], x["k"].permute(1, 0, 2)[None],
                             x["v"].permute(1, 0, 2)[None], x["q_descale"], x["k_descale"],
                             x["v_descale"], 0.1, True)
    for name in ("o", "bound", "pv_abs"):
        assert np.allclose(r[name], f[name][0].transpose(1, 0, 2), rtol=1e-12, atol=1e-14), name
    assert np.allclose(r["lse"], f["lse"][0], rtol=1e-12, atol=1e-12)
