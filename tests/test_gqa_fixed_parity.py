"""Fixed-length [B, H, Nq, d] attention with grouped key/value heads [B, Hkv, Nk, d] and
Nq != Nk (fa_fwd_gqa, fa_bwd_gqa, reached through fa.forward / fa.backward when k's heads or
length differ from q's): against the fp64 oracle, and bit for bit against the packed path on
the same values (same arithmetic, other addressing)."""
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import random_varlen
from tests.gpu_util import check_grads
from tests.test_varlen_parity import check_fwd_with_empty_rows

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Hkv, Nq, Nk
    (2, 8, 2, 300, 300),      # GQA, square
    (1, 4, 1, 129, 700),      # MQA, a chunk of queries against a longer history
    (3, 2, 2, 257, 100),      # more queries than keys: early rows see no key when causal
    (1, 6, 3, 1, 1000),       # one query
]


def to_bhsd(t, B, N):
    """[B*N, heads, d] (packed, equal lengths) -> [B, heads, N, d]."""
    return t.reshape(B, N, t.shape[1], t.shape[2]).transpose(1, 2).contiguous()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", CASES)
def test_grouped_fixed_length_against_oracle_and_packed_path(case, d, causal):
    B, H, Hkv, Nq, Nk = case
    x = random_varlen([Nq] * B, [Nk] * B, H, Hkv, d, seed=B * 100 + Nq + d + causal)
    scale = d ** -0.5
    q, k, v, do = (to_bhsd(x[n], B, Nq if n in ("q", "do") else Nk).cuda()
                   for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, scale=scale, causal=causal)
    fa.fa_device_status()
    ref = oracle.attention_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], scale, causal,
                                  do=x["do"])
    # the oracle is packed: bring the library's results to the packed layout
    pk = lambda t: t.transpose(1, 2).reshape(-1, t.shape[1], t.shape[3])  # noqa: E731
    got = {"o": pk(o), "lse": lse.permute(1, 0, 2).reshape(H, B * Nq), "dq": pk(dq),
           "dk": pk(dk), "dv": pk(dv)}
    what = f"B={B} H={H} Hkv={Hkv} Nq={Nq} Nk={Nk} d={d} causal={causal}"
    check_fwd_with_empty_rows(got, ref, what)
    check_grads(got, ref, torch.bfloat16, what)
    # the packed path on the same values
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "do", "cu_q", "cu_k")}
    o2, lse2 = fa.forward_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], Nq, Nk,
                                 scale=scale, causal=causal)
    g2 = fa.backward_varlen(dev["q"], dev["k"], dev["v"], o2, dev["do"], lse2, dev["cu_q"],
                            dev["cu_k"], Nq, Nk, scale=scale, causal=causal)
    fa.fa_device_status()
    assert torch.equal(got["o"], o2) and torch.equal(got["lse"], lse2)
    for a, b in zip((got["dq"], got["dk"], got["dv"]), g2):
        assert torch.equal(a, b)
