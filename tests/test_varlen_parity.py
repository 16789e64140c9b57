"""Parity of the packed variable-length entry points (fa_fwd_varlen, fa_bwd_varlen) against the
fp64 oracle: ragged sequences, grouped key/value heads (GQA, MQA), more keys than queries
(chunked prefill, bottom-right causal mask), more queries than keys (rows that see no key),
empty sequences; bitwise agreement with the fixed-length entry points on equal-length batches;
outputs confined to their buffers; determinism."""
import numpy as np
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import random_qkv, random_varlen
from tests.gpu_util import check_fwd, check_grads, f64, guarded_empty

pytestmark = pytest.mark.gpu

CASES = {
    # name: (query lengths, key lengths, H, Hkv)
    "square_mha": ([1, 130, 257, 64, 300], [1, 130, 257, 64, 300], 4, 4),
    "square_gqa": ([129, 1, 383], [129, 1, 383], 8, 2),
    "mqa": ([200, 77], [200, 77], 4, 1),
    "chunked_prefill": ([100, 128, 1, 300], [400, 128, 77, 429], 4, 2),
    "more_queries_than_keys": ([300, 50, 260], [100, 50, 3], 2, 1),
    "empty_sequences": ([0, 5, 130, 7], [10, 0, 130, 0], 2, 2),
}


def run_varlen(x, causal, scale):
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "do", "cu_q", "cu_k")}
    o, lse = fa.forward_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], x["max_q"],
                               x["max_k"], scale=scale, causal=causal)
    dq, dk, dv = fa.backward_varlen(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, dev["cu_q"],
                                    dev["cu_k"], x["max_q"], x["max_k"], scale=scale,
                                    causal=causal)
    fa.fa_device_status()
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def check_fwd_with_empty_rows(got, ref, what):
    """Rows that see no key: O exactly 0 and lse -inf on both sides; the rest within the bf16
    bounds of the fixed-length tests."""
    lse, lse_ref = f64(got["lse"]), ref["lse"]            # [H, total_q]
    o, o_ref = f64(got["o"]), ref["o"]                    # [total_q, H, d]
    empty = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == empty).all(), f"-inf rows differ {what}"
    assert (o[empty.T] == 0.0).all(), f"rows without keys are not 0 {what}"
    if (~empty).any():
        return check_fwd(o[~empty.T], lse[~empty], o_ref[~empty.T], lse_ref[~empty],
                         torch.bfloat16, what)
    return {}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", list(CASES))
def test_varlen_against_oracle(case, d, causal):
    lens_q, lens_k, H, Hkv = CASES[case]
    x = random_varlen(lens_q, lens_k, H, Hkv, d, seed=len(case) * 7 + d + causal)
    scale = d ** -0.5
    got = run_varlen(x, causal, scale)
    ref = oracle.attention_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], scale, causal,
                                  do=x["do"])
    what = f"{case} d={d} causal={causal}"
    stats = check_fwd_with_empty_rows(got, ref, what)
    gstats = check_grads(got, ref, torch.bfloat16, what)
    print(what, stats, gstats)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_equal_lengths_match_fixed_layout_bit_for_bit(d, causal):
    """cu = [0, N, 2N, ...] with Hkv = H is the fixed-length problem in token-major order: the
    same tiles and the same arithmetic, so every output agrees exactly."""
    B, H, N = 3, 2, 333
    x = random_qkv(B, H, N, d, seed=77 + d)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=causal)
    pk = lambda t: t.transpose(1, 2).reshape(B * N, H, d).contiguous()  # noqa: E731
    cu = torch.arange(0, B * N + 1, N, dtype=torch.int32, device="cuda")
    o2, lse2 = fa.forward_varlen(pk(q), pk(k), pk(v), cu, cu, N, N, causal=causal)
    dq2, dk2, dv2 = fa.backward_varlen(pk(q), pk(k), pk(v), o2, pk(do), lse2, cu, cu, N, N,
                                       causal=causal)
    fa.fa_device_status()
    assert torch.equal(o2, pk(o))
    assert torch.equal(lse2, lse.permute(1, 0, 2).reshape(H, B * N))
    for a, b in ((dq2, dq), (dk2, dk), (dv2, dv)):
        assert torch.equal(a, pk(b))


def test_varlen_outputs_stay_inside_their_buffers_and_are_deterministic():
    lens_q, lens_k, H, Hkv, d = [0, 5, 130, 300], [10, 0, 130, 129], 4, 2, 128
    x = random_varlen(lens_q, lens_k, H, Hkv, d, seed=5)
    q, k, v, do, cu_q, cu_k = (x[n].cuda() for n in ("q", "k", "v", "do", "cu_q", "cu_k"))
    tq, tk = q.shape[0], k.shape[0]
    for causal in (False, True):
        outs = []
        for _ in range(2):
            o, co = guarded_empty((tq, H, d), torch.bfloat16)
            lse, cl = guarded_empty((H, tq), torch.float32)
            fa.fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, x["max_q"], x["max_k"], d ** -0.5,
                             causal)
            dq, cq = guarded_empty((tq, H, d), torch.bfloat16)
            dk, ck = guarded_empty((tk, Hkv, d), torch.bfloat16)
            dv, cv = guarded_empty((tk, Hkv, d), torch.bfloat16)
            ws, cw = guarded_empty((fa.fa_bwd_varlen_workspace_bytes(tq, H, d),), torch.uint8)
            fa.fa_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_q, cu_k, x["max_q"], x["max_k"],
                             d ** -0.5, causal, ws)
            fa.fa_device_status()
            for c in (co, cl, cq, ck, cv, cw):
                c()
            outs.append([t.clone() for t in (o, lse, dq, dk, dv)])
        for a, b in zip(*outs):
            assert torch.equal(a, b), "packed path is not bit-for-bit deterministic"


def test_max_seqlen_larger_than_needed_only_adds_idle_blocks():
    """max_seqlen is an upper bound: a generous one gives the same result."""
    x = random_varlen([70, 260], [300, 260], 4, 2, 64, seed=9)
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "cu_q", "cu_k")}
    a = fa.forward_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], 260, 300,
                          causal=True)
    b = fa.forward_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], 1000, 1000,
                          causal=True)
    fa.fa_device_status()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_chunked_prefill_gqa_at_size_sampled_heads():
    """Llama-style grouping (32 query heads over 8 key/value heads, d = 128) on sequences of a
    few thousand tokens, with query chunks shorter than their key sequences; the oracle checks
    every query head of two key/value groups (so dK and dV sum over complete groups)."""
    lens_q, lens_k, H, Hkv, d = [2048, 512, 1500], [2048, 4096, 1500], 32, 8, 128
    x = random_varlen(lens_q, lens_k, H, Hkv, d, seed=11)
    got = run_varlen(x, True, d ** -0.5)
    G = H // Hkv
    groups = [0, 5]
    heads = [h for hk in groups for h in range(hk * G, (hk + 1) * G)]
    ref = oracle.attention_varlen(x["q"][:, heads], x["k"][:, groups], x["v"][:, groups],
                                  x["cu_q"], x["cu_k"], d ** -0.5, True, do=x["do"][:, heads])
    sub = {"o": got["o"][:, heads], "lse": got["lse"][heads], "dq": got["dq"][:, heads],
           "dk": got["dk"][:, groups], "dv": got["dv"][:, groups]}
    stats = check_fwd(sub["o"], sub["lse"], ref["o"], ref["lse"], torch.bfloat16, "prefill")
    gstats = check_grads(sub, ref, torch.bfloat16, "prefill")
    print("chunked prefill GQA", stats, gstats)
