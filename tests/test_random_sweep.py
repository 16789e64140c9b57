"""Seeded random sweep over packed-batch problems: per case a random number of sequences with
random query and key lengths (including empty, single-token and ragged ones, more keys than
queries and the reverse), a random head grouping, d, mask and decode split count.  Every
case runs the packed forward and backward and, where its shape allows, the split-KV decode,
each checked against the fp64 oracle with the bf16 tolerances of the fixed-length tests."""
import os

import numpy as np
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import random_varlen
from tests.gpu_util import check_grads
from tests.test_varlen_parity import check_fwd_with_empty_rows

pytestmark = pytest.mark.gpu

# FA_SWEEP_CASES / FA_SWEEP_FIXED_CASES widen the sweep for a longer stress run
N_CASES = int(os.environ.get("FA_SWEEP_CASES", "48"))
N_FIXED_CASES = int(os.environ.get("FA_SWEEP_FIXED_CASES", "16"))


def draw_case(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 6))
    Hkv = int(rng.choice([1, 2, 4]))
    H = Hkv * int(rng.choice([1, 2, 3, 4]))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))

    def length(hi):
        kind = rng.random()
        if kind < 0.1:
            return 0
        if kind < 0.2:
            return 1
        return int(rng.integers(2, hi))

    lens_k = [length(700) for _ in range(B)]
    # queries: a chunk of the keys (chunked prefill), the same length, or longer
    lens_q = []
    for nk in lens_k:
        mode = rng.random()
        if mode < 0.4:
            lens_q.append(int(rng.integers(0, nk + 1)))
        elif mode < 0.8:
            lens_q.append(nk)
        else:
            lens_q.append(nk + int(rng.integers(1, 200)))
    if max(lens_q) == 0:
        lens_q[0] = 1
    if max(lens_k) == 0:
        lens_k[0] = 1
    splits = int(rng.integers(1, 9))
    return lens_q, lens_k, H, Hkv, d, causal, splits


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_packed_problem(seed):
    lens_q, lens_k, H, Hkv, d, causal, splits = draw_case(1000 + seed)
    what = f"seed={seed} lens_q={lens_q} lens_k={lens_k} H={H} Hkv={Hkv} d={d} causal={causal}"
    x = random_varlen(lens_q, lens_k, H, Hkv, d, seed=seed)
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "do", "cu_q", "cu_k")}
    scale = d ** -0.5
    o, lse = fa.forward_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], x["max_q"],
                               x["max_k"], scale=scale, causal=causal)
    dq, dk, dv = fa.backward_varlen(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, dev["cu_q"],
                                    dev["cu_k"], x["max_q"], x["max_k"], scale=scale,
                                    causal=causal)
    fa.fa_device_status()
    ref = oracle.attention_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], scale, causal,
                                  do=x["do"])
    check_fwd_with_empty_rows({"o": o, "lse": lse}, ref, what)
    got = {"dq": dq, "dk": dk, "dv": dv}
    if sum(lens_q) and sum(lens_k):
        check_grads(got, ref, torch.bfloat16, what)
    if x["max_q"] <= 128:  # the decode kernel takes up to 128 queries per sequence
        od, lsed = fa.forward_decode(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"],
                                     x["max_q"], x["max_k"], scale=scale, causal=causal,
                                     num_splits=splits)
        fa.fa_device_status()
        check_fwd_with_empty_rows({"o": od, "lse": lsed}, ref, what + f" decode splits={splits}")


@pytest.mark.parametrize("seed", range(N_FIXED_CASES))
def test_random_fixed_length_problem(seed):
    """Fixed-length [B, H, N, d] calls with random sizes, masks and scales (including
    non-standard ones), against the oracle.  Inputs stay at most N(0,1) in magnitude: the
    absolute bf16 bound on O (1.5e-2) presumes |V| of that size (one bf16 ulp of an output of
    magnitude 2-4 is already 1.6e-2)."""
    from exact_attention_25_gb300.inputs import random_qkv

    rng = np.random.default_rng(5000 + seed)
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    N = int(rng.integers(1, 900))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    scale = float(rng.choice([d ** -0.5, 0.02, 0.3, -0.1]))
    x = random_qkv(B, H, N, d, seed=seed, in_scale=float(rng.choice([0.5, 1.0])))
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, scale=scale, causal=causal)
    fa.fa_device_status()
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal)
    what = f"seed={seed} B={B} H={H} N={N} d={d} causal={causal} scale={scale}"
    from tests.gpu_util import check_fwd

    check_fwd(o, lse, ref["o"], ref["lse"], torch.bfloat16, what, check_mean=N > 1)
    check_grads({"dq": dq, "dk": dk, "dv": dv}, ref, torch.bfloat16, what)


@pytest.mark.parametrize("seed", range(max(1, N_CASES // 4)))
def test_random_packed_e4m3_problem(seed):
    """The packed e4m3 forward on the same kind of random batches (d = 128), within the
    oracle's per-element rounding bound."""
    from exact_attention_25_gb300.inputs import random_fp8_varlen

    lens_q, lens_k, H, Hkv, _, causal, _ = draw_case(7000 + seed)
    x = random_fp8_varlen(lens_q, lens_k, H, Hkv, 128, seed=seed,
                          in_scale=float(np.random.default_rng(seed).choice([0.3, 1.0, 3.0])))
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "cu_q", "cu_k")}
    scale = 128 ** -0.5
    o, lse = fa.forward_fp8_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"],
                                   x["max_q"], x["max_k"], x["q_descale"], x["k_descale"],
                                   x["v_descale"], scale=scale, causal=causal)
    fa.fa_device_status()
    r = oracle.attention_fp8_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"],
                                    x["q_descale"], x["k_descale"], x["v_descale"], scale, causal)
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    tol = r["bound"] + 2.0 ** -8 * (np.abs(r["o"]) + r["bound"]) + 1e-4 * r["pv_abs"] + 1e-6
    what = f"seed={seed} lens_q={lens_q} lens_k={lens_k} H={H} Hkv={Hkv} causal={causal}"
    assert np.all(np.abs(o - r["o"]) <= tol), what
    assert np.array_equal(np.isneginf(lse), np.isneginf(r["lse"])), what
    fin = np.isfinite(r["lse"])
    assert np.abs(lse[fin] - r["lse"][fin]).max(initial=0.0) <= 1e-3, what
