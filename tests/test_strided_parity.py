"""Strided packed tensors (fa_fwd_varlen_strided, fa_bwd_varlen_strided through the Python
binding): q, k and v as views of one fused projection, outputs and gradients written into
views of fused buffers.  Only the addressing differs from contiguous tensors, so every result
must agree with the contiguous call bit for bit, and nothing outside the views may change."""
import pytest
import torch

import exact_attention_25_gb300 as fa
from exact_attention_25_gb300.inputs import random_varlen

pytestmark = pytest.mark.gpu


def fused(x, H, Hkv):
    """One [total, H + 2 Hkv, d] buffer holding q, k, v side by side per token (the output of
    a fused QKV projection with grouped K/V heads); returns the buffer and the three views."""
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    buf = torch.cat([q, k, v], dim=1).contiguous()
    return buf, buf[:, :H], buf[:, H:H + Hkv], buf[:, H + Hkv:]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 2)])
def test_fused_qkv_views_match_contiguous_bit_for_bit(H, Hkv, d, causal):
    lens = [130, 1, 257]
    x = random_varlen(lens, lens, H, Hkv, d, seed=H * 10 + d + causal)
    buf, qv, kv, vv = fused(x, H, Hkv)
    assert not qv.is_contiguous() and qv.stride() == (buf.stride(0), d, 1)
    cu = x["cu_q"].cuda()
    n = max(lens)
    q, k, v, do = (x[t].cuda() for t in ("q", "k", "v", "do"))
    o_ref, lse_ref = fa.forward_varlen(q, k, v, cu, cu, n, n, causal=causal)
    g_ref = fa.backward_varlen(q, k, v, o_ref, do, lse_ref, cu, cu, n, n, causal=causal)

    # outputs into views of fused buffers: O into half of a [total, H, 2d] buffer, the
    # gradients into one fused [total, H + 2 Hkv, d] buffer like the projection's
    T = q.shape[0]
    obuf = torch.full((T, H, 2 * d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ov = obuf[:, :, :d]
    lse = torch.empty((H, T), dtype=torch.float32, device="cuda")
    fa.fa_fwd_varlen(qv, kv, vv, ov, lse, cu, cu, n, n, d ** -0.5, causal)
    gbuf = torch.full((T, H + 2 * Hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dqv, dkv, dvv = gbuf[:, :H], gbuf[:, H:H + Hkv], gbuf[:, H + Hkv:]
    ws = torch.empty(fa.fa_bwd_varlen_workspace_bytes(T, H, d), dtype=torch.uint8, device="cuda")
    dobuf = torch.cat([do, torch.zeros_like(do)], dim=2)  # dO as a strided view as well
    fa.fa_bwd_varlen(qv, kv, vv, ov, dobuf[:, :, :d], lse, dqv, dkv, dvv, cu, cu, n, n,
                     d ** -0.5, causal, ws)
    fa.fa_device_status()
    assert torch.equal(ov, o_ref) and torch.equal(lse, lse_ref)
    assert torch.isnan(obuf[:, :, d:].float()).all(), "write outside the O view"
    for got, ref in zip((dqv, dkv, dvv), g_ref):
        assert torch.equal(got, ref)
    assert not torch.isnan(gbuf.float()).any(), "a gradient view was not fully written"


def test_unsupported_views_are_rejected():
    x = random_varlen([64], [64], 2, 2, 64, seed=2)
    q, k, v = (x[t].cuda() for t in ("q", "k", "v"))
    cu = x["cu_q"].cuda()
    o = torch.empty_like(q)
    qt = q.transpose(0, 1).contiguous().transpose(0, 1)  # head-major storage: head step > row step
    with pytest.raises(fa.FaError) as ei:
        fa.fa_fwd_varlen(qt, k, v, o, None, cu, cu, 64, 64, 0.125, False)
    assert ei.value.code == -1
    with pytest.raises(ValueError):
        fa.fa_fwd_varlen(q[:, :, ::2], k, v, o, None, cu, cu, 64, 64, 0.125, False)
