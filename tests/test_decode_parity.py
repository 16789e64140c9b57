"""Parity of the split-KV decode entry point (fa_fwd_decode) against the fp64 oracle: one or a
few queries per sequence (speculative decoding under the causal mask) against key histories
from 1 to thousands of keys, grouped heads G = 1..16 packed into one tile, split counts from 1
to more than the sequence has blocks, empty sequences; outputs confined to their buffers,
determinism, and a decode step at serving size."""
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import random_varlen
from tests.gpu_util import check_fwd, f64, guarded_empty
from tests.test_varlen_parity import check_fwd_with_empty_rows

pytestmark = pytest.mark.gpu


def run_decode(x, causal, splits, scale):
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "cu_q", "cu_k")}
    o, lse = fa.forward_decode(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], x["max_q"],
                               x["max_k"], scale=scale, causal=causal, num_splits=splits)
    fa.fa_device_status()
    return {"o": o, "lse": lse}


CASES = {
    # name: (query lengths, key lengths, H, Hkv)
    "one_token_mha": ([1, 1, 1], [1, 127, 1000], 4, 4),
    "one_token_gqa8": ([1, 1, 1, 1], [129, 128, 2000, 5], 32, 4),
    "one_token_mqa16": ([1, 1], [700, 3000], 16, 1),
    "speculative_4": ([4, 4, 2], [300, 1025, 2], 16, 2),
    "full_tile": ([16, 9], [16, 900], 8, 1),
    "empty_sequences": ([1, 0, 1, 1], [0, 50, 260, 1], 8, 2),
    "heads_over_two_tiles": ([8, 3], [700, 129], 32, 1),      # 32 x 8 rows: chunks of 16 heads
    "group_not_a_power_of_two": ([11, 5], [300, 1000], 12, 1),  # 12 x 11 rows: chunks of 6
}


@pytest.mark.parametrize("splits", [1, 2, 3, 8, 9, 16])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", list(CASES))
def test_decode_against_oracle(case, d, causal, splits):
    lens_q, lens_k, H, Hkv = CASES[case]
    x = random_varlen(lens_q, lens_k, H, Hkv, d, seed=3 * len(case) + d + splits, with_do=False)
    scale = d ** -0.5
    got = run_decode(x, causal, splits, scale)
    ref = oracle.attention_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], scale, causal)
    print(case, d, causal, splits, check_fwd_with_empty_rows(got, ref, f"{case} s={splits}"))


@pytest.mark.parametrize("causal", [False, True])
def test_decode_agrees_with_the_varlen_forward(causal):
    """Same problem through fa_fwd_varlen: both within bf16 rounding of each other."""
    x = random_varlen([1, 3, 1], [4000, 777, 129], 32, 8, 128, seed=17, with_do=False)
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "cu_q", "cu_k")}
    a = run_decode(x, causal, 5, 128 ** -0.5)
    o, lse = fa.forward_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], x["max_q"],
                               x["max_k"], causal=causal)
    fa.fa_device_status()
    assert (a["o"].float() - o.float()).abs().max().item() <= 1.6e-2
    assert (a["lse"] - lse).abs().max().item() <= 1e-3


def test_decode_outputs_stay_inside_their_buffers_and_are_deterministic():
    lens_q, lens_k, H, Hkv, d = [1, 0, 4, 1], [300, 20, 1000, 0], 8, 2, 128
    x = random_varlen(lens_q, lens_k, H, Hkv, d, seed=8, with_do=False)
    q, k, v, cu_q, cu_k = (x[n].cuda() for n in ("q", "k", "v", "cu_q", "cu_k"))
    tq = q.shape[0]
    for splits in (1, 4, 16):  # one range, merged in the kernel, merged by the combine kernel
        outs = []
        for _ in range(2):
            o, co = guarded_empty((tq, H, d), torch.bfloat16)
            lse, cl = guarded_empty((H, tq), torch.float32)
            nbytes = fa.fa_decode_workspace_bytes(tq, H, d, splits)
            ws, cw = guarded_empty((max(nbytes, 16),), torch.uint8)
            fa.fa_fwd_decode(q, k, v, o, lse, cu_q, cu_k, x["max_q"], x["max_k"], d ** -0.5, True,
                             splits, ws if nbytes else None)
            fa.fa_device_status()
            for c in (co, cl, cw):
                c()
            outs.append((o.clone(), lse.clone()))
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_decode_step_at_serving_size_sampled_groups():
    """A decode step of 8 sequences (one new token each, 32 query heads over 8 key/value heads,
    d = 128) against key histories of 3 K to 16 K tokens, with the suggested split count; the
    oracle checks every query head of two groups."""
    lens_k = [16384, 3000, 9000, 12000, 4096, 16000, 7777, 10000]
    lens_q, H, Hkv, d = [1] * len(lens_k), 32, 8, 128
    x = random_varlen(lens_q, lens_k, H, Hkv, d, seed=23, with_do=False)
    splits = fa.fa_decode_num_splits(len(lens_k), Hkv, max(lens_k))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert splits == fa.load().fa_decode_splits_for(len(lens_k), Hkv, max(lens_k), sms) >= 1
    got = run_decode(x, True, splits, d ** -0.5)
    G = H // Hkv
    groups = [1, 6]
    heads = [h for hk in groups for h in range(hk * G, (hk + 1) * G)]
    ref = oracle.attention_varlen(x["q"][:, heads], x["k"][:, groups], x["v"][:, groups],
                                  x["cu_q"], x["cu_k"], d ** -0.5, True)
    stats = check_fwd(f64(got["o"])[:, heads], f64(got["lse"])[heads], ref["o"], ref["lse"],
                      torch.bfloat16, "decode at size")
    print("decode at size, splits", splits, stats)


def test_decode_rejects_more_queries_than_one_tile():
    x = random_varlen([129], [300], 2, 1, 64, seed=1, with_do=False)  # 129 queries > 128 rows
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "cu_q", "cu_k")}
    with pytest.raises(fa.FaError) as ei:
        fa.forward_decode(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], 129, 300,
                          num_splits=1)
    assert ei.value.code == -1
