"""Long ragged sequences (N = 8191 and 32001, one short of / one past a multiple of every tile
size), forward and backward, against the fp64 oracle on sampled rows: the first rows, rows of
the ragged last block, and rows in between; dK / dV on a few key rows including the last."""
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import random_qkv
from tests.gpu_util import TOL_GRAD_REL_L2, check_fwd, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(8191, 128), (8191, 64), (32001, 128)])
def test_long_ragged_sequence_sampled_rows(N, d, causal):
    x = random_qkv(1, 2, N, d, seed=N + d + causal)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=causal)
    fa.fa_device_status()
    last_block = N - N % 128
    rows = sorted({0, 1, 127, 128, N // 2, last_block - 1, last_block, N - 2, N - 1})
    krows = [0, N - 1] if N < 10000 else [N - 1]
    h = 1
    ref = oracle.attention_rows_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], x["do"][0, h],
                                     d ** -0.5, causal, rows, krows)
    what = f"N={N} d={d} causal={causal}"
    check_fwd(o[0, h, rows], lse[0, h, rows], ref["o"], ref["lse"], torch.bfloat16, what,
              check_mean=False)
    assert rel_l2(dq[0, h, rows], ref["dq"]) <= TOL_GRAD_REL_L2, what
    assert rel_l2(dk[0, h, krows], ref["dk"]) <= TOL_GRAD_REL_L2, what
    assert rel_l2(dv[0, h, krows], ref["dv"]) <= TOL_GRAD_REL_L2, what
