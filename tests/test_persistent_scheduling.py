"""The tensor-core kernels run persistently: a CTA takes the tiles of CTAs that have not started
yet (cluster launch control) and walks them in the grouped heaviest-first order.  These cases
make every CTA walk many short tiles - more heads than SMs, one- and two-block tiles, tiles
without keys, ragged tails, grouped heads and packed batches - and compare against the fp64
oracle; and since the order in which CTAs take tiles can change from run to run, repeated runs
must agree bit for bit."""
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import random_qkv, random_varlen
from tests.gpu_util import check_fwd, check_grads
from tests.test_varlen_parity import check_fwd_with_empty_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N", [(4, 96, 129), (2, 160, 300), (8, 40, 257)])
def test_many_short_tiles_per_cta(B, H, N, d, causal):
    """B * H heads well above the 152 SMs, each of 1-3 blocks: every CTA runs several tiles
    of several heads, across head groups (under the causal mask) and the ragged last block."""
    x = random_qkv(B, H, N, d, seed=B * 1000 + H + N + d + causal)
    q, k, v, do = (t.cuda() for t in (x["q"], x["k"], x["v"], x["do"]))
    scale = d ** -0.5
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, scale=scale, causal=causal)
    fa.fa_device_status()
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal)
    what = f"B={B} H={H} N={N} d={d} causal={causal}"
    check_fwd(o.cpu(), lse.cpu(), ref["o"], ref["lse"], torch.bfloat16, what)
    check_grads({"dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}, ref, torch.bfloat16, what)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_batch_with_empty_and_keyless_tiles(causal):
    """A packed batch whose grid (sized by the longest sequence) holds many tiles beyond the
    shorter sequences, and sequences with more queries than keys (tiles without keys under the
    causal mask): all roles of a CTA must skip the same tiles."""
    lens_q = [1, 300, 0, 129, 257, 40, 128, 2] * 6
    lens_k = [200, 64, 17, 129, 100, 40, 0, 700] * 6
    H, Hkv, d = 8, 2, 128
    x = random_varlen(lens_q, lens_k, H, Hkv, d, seed=31 + causal)
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "do", "cu_q", "cu_k")}
    mq, mk = max(lens_q), max(lens_k)
    o, lse = fa.forward_varlen(dev["q"], dev["k"], dev["v"], dev["cu_q"], dev["cu_k"], mq, mk,
                               scale=0.09, causal=causal)
    dq, dk, dv = fa.backward_varlen(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, dev["cu_q"],
                                    dev["cu_k"], mq, mk, scale=0.09, causal=causal)
    fa.fa_device_status()
    ref = oracle.attention_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], 0.09, causal,
                                  do=x["do"])
    got = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    check_fwd_with_empty_rows(got, ref, f"packed causal={causal}")
    check_grads(got, ref, torch.bfloat16, f"packed causal={causal}")


def test_repeated_runs_agree_bit_for_bit_whatever_the_tile_hand_out():
    """Each tile's arithmetic does not depend on which CTA runs it or when, so forward and
    backward results are identical across runs, including when another kernel occupies part of
    the GPU meanwhile (a concurrent stream changes which CTAs take which tiles)."""
    x = random_qkv(2, 64, 700, 128, seed=77)
    q, k, v, do = (t.cuda() for t in (x["q"], x["k"], x["v"], x["do"]))
    first = None
    side = torch.cuda.Stream()
    big = torch.randn(4096, 4096, device="cuda")
    for run in range(4):
        if run >= 2:  # keep some SMs busy on another stream while the kernels run
            with torch.cuda.stream(side):
                for _ in range(4):
                    big = big @ big.t() * 1e-4
        o, lse = fa.forward(q, k, v, causal=True)
        dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=True)
        fa.fa_device_status()
        torch.cuda.synchronize()
        outs = [t.clone() for t in (o, lse, dq, dk, dv)]
        if first is None:
            first = outs
        else:
            for a, b, n in zip(first, outs, ("o", "lse", "dq", "dk", "dv")):
                assert torch.equal(a, b), (run, n)
