"""Stream order around the kernels launched as programmatic dependents: the backward's dK/dV
and dQ kernels (dQ may start in the tail of dK/dV) and the decode's split kernel.  Work queued
on the same stream right before a call, with no synchronisation in between, must be complete
before the call reads its inputs; work queued right after it must not start before every kernel
of the call has completed.  Each case produces the inputs with torch kernels immediately before
the call, overwrites every input (and the workspace) immediately after it, and compares the
outputs bit for bit with the same call run between device synchronisations: the kernels are
deterministic, so any read of a half-written or already-overwritten input would show."""
import pytest
import torch

import exact_attention_25_gb300 as fa
from exact_attention_25_gb300.inputs import random_qkv

pytestmark = pytest.mark.gpu


def _pristine(B, H, N, d, seed, Hkv=None):
    x = random_qkv(B, H, N, d, seed=seed)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    if Hkv is not None:  # grouped heads: keep the first Hkv key/value heads
        k, v = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    return q, k, v, do


def _reference_backward(q, k, v, do, causal):
    torch.cuda.synchronize()
    o, lse = fa.forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=causal)
    torch.cuda.synchronize()
    return o, lse, (dq, dk, dv)


def _spoil(*ts):
    for t in ts:
        t.fill_(float("nan") if t.is_floating_point() else 0xFF)


@pytest.mark.parametrize("B,H,Hkv,N,d,causal", [
    (2, 4, None, 1536, 128, True),
    (1, 6, None, 1000, 64, False),
    (2, 4, 2, 1100, 128, True),
])
def test_backward_sees_inputs_queued_before_and_is_done_before_what_follows(B, H, Hkv, N, d,
                                                                           causal):
    q0, k0, v0, do0 = _pristine(B, H, N, d, seed=900 + N, Hkv=Hkv)
    o0, lse0, ref = _reference_backward(q0, k0, v0, do0, causal)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    for rep in range(3):
        torch.cuda.synchronize()
        # inputs written by torch kernels queued right before the call
        q, k, v, do, o, lse = (t.clone() for t in (q0, k0, v0, do0, o0, lse0))
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, q.shape[-1] ** -0.5, causal, ws)
        # and overwritten by kernels queued right after it, with the workspace
        _spoil(q, k, v, do, o, lse, ws)
        torch.cuda.synchronize()
        for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            assert torch.equal(got, want), (rep, name)


@pytest.mark.parametrize("order", [(0, 1, 2), (0, 2, 1)])
def test_backward_stages_queued_back_to_back_in_either_order(order):
    B, H, N, d, causal = 2, 4, 1300, 128, True
    q0, k0, v0, do0 = _pristine(B, H, N, d, seed=77)
    o0, lse0, ref = _reference_backward(q0, k0, v0, do0, causal)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    q, k, v, do, o, lse = (t.clone() for t in (q0, k0, v0, do0, o0, lse0))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for stage in order:
        fa.fa_bwd_stage(q, k, v, o, do, lse, dq, dk, dv, d ** -0.5, causal, ws, stage)
    _spoil(q, k, v, do, o, lse, ws)
    torch.cuda.synchronize()
    for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        assert torch.equal(got, want), (order, name)


def test_two_backward_calls_share_a_workspace_back_to_back():
    B, H, N, d = 1, 8, 2048, 128
    a = _pristine(B, H, N, d, seed=11)
    b = _pristine(B, H, N, d, seed=12)
    oa, la, ref_a = _reference_backward(*a, True)
    ob, lb, ref_b = _reference_backward(*b, False)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    outs = []
    for (q, k, v, do), o, lse, causal in ((a, oa, la, True), (b, ob, lb, False)):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, d ** -0.5, causal, ws)
        outs.append((dq, dk, dv))
    torch.cuda.synchronize()
    for got3, want3 in zip(outs, (ref_a, ref_b)):
        for got, want in zip(got3, want3):
            assert torch.equal(got, want)


def test_decode_sees_inputs_queued_before_and_is_done_before_what_follows():
    B, H, Hkv, d, nk = 4, 16, 4, 128, 3000
    g = torch.Generator().manual_seed(5)
    q0 = torch.randn(B, H, d, generator=g).to(torch.bfloat16).cuda()
    k0 = torch.randn(B * nk, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    v0 = torch.randn(B * nk, Hkv, d, generator=g).to(torch.bfloat16).cuda()
    cu_q = torch.arange(0, B + 1, dtype=torch.int32).cuda()
    cu_k = (torch.arange(0, B + 1, dtype=torch.int32) * nk).cuda()
    splits = 6
    nbytes = fa.fa_decode_workspace_bytes(B, H, d, splits)
    torch.cuda.synchronize()
    ref_o, ref_l = fa.forward_decode(q0, k0, v0, cu_q, cu_k, 1, nk, num_splits=splits)
    torch.cuda.synchronize()
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for rep in range(3):
        torch.cuda.synchronize()
        q, k, v = q0.clone(), k0.clone(), v0.clone()
        o = torch.empty_like(q)
        lse = torch.empty((H, B), dtype=torch.float32, device="cuda")
        fa.fa_fwd_decode(q, k, v, o, lse, cu_q, cu_k, 1, nk, d ** -0.5, False, splits, ws)
        _spoil(q, k, v, ws)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o), rep
        assert torch.equal(lse, ref_l), rep
