"""The bounds-checked library (libfa_checked.so, built with FA_CHECKED): every element the
kernels read or write directly in global memory is tested against its buffer's extent, an
access outside it is skipped and reported as FA_ERR_OUT_OF_BOUNDS.

  * On well-formed calls it gives the regular library's results bit for bit and reports
    nothing.
  * With malformed cu_seqlens (not monotonic, negative, past the packed total, sequences
    longer than max_seqlen) the kernels clamp every sequence to the packed tensors, so the
    checks report nothing and guard regions around every output stay untouched.
  * With the test hook that takes every extent one row step short, the checks must fire: the
    call reports FA_ERR_OUT_OF_BOUNDS and the accesses past the shortened extent are skipped.
"""
import os

import pytest
import torch

import exact_attention_25_gb300 as fa
from exact_attention_25_gb300 import _lib
from exact_attention_25_gb300.inputs import random_qkv, random_varlen

pytestmark = pytest.mark.gpu

SHRINK_EXTENTS = 2  # fa_debug_set_flags value of the one-row-step-short hook
PAD = 7             # guard rows before and after every packed output


@pytest.fixture(scope="module")
def checked():
    if not os.path.exists(_lib.LIB_CHECKED_PATH):
        from exact_attention_25_gb300 import build

        build.build(checked=True)
    with _lib.library(_lib.LIB_CHECKED_PATH) as lib:
        assert fa.fa_checked_build()
        lib.fa_debug_set_flags(0)
        yield lib
        lib.fa_debug_set_flags(0)


def guarded(shape, dtype):
    """A NaN-filled buffer with PAD guard rows on both sides of dim 0 and the inner view."""
    buf = torch.full((shape[0] + 2 * PAD, *shape[1:]), float("nan"), dtype=dtype, device="cuda")
    return buf, buf[PAD:PAD + shape[0]]


def guarded_lse(H, T):
    """[H, T] statistics inside a flat NaN buffer with guards before and after."""
    flat = torch.full((H * T + 2 * 64,), float("nan"), dtype=torch.float32, device="cuda")
    return flat, flat[64:64 + H * T].view(H, T)


def assert_guards_intact(buf, what):
    head, tail = buf[:PAD].float(), buf[buf.shape[0] - PAD:].float()
    assert torch.isnan(head).all() and torch.isnan(tail).all(), f"{what}: write outside the buffer"


def assert_flat_guards_intact(flat, what):
    assert torch.isnan(flat[:64]).all() and torch.isnan(flat[-64:]).all(), what


def run_packed(x, cu_q, cu_k, max_q, max_k, causal, splits):
    """Forward, backward and split-KV decode into guarded buffers; returns the results and
    checks that nothing outside the outputs changed."""
    H, d = x["q"].shape[1], x["q"].shape[2]
    Hkv = x["k"].shape[1]
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    Tq, Tk = q.shape[0], k.shape[0]
    scale = d ** -0.5
    obuf, o = guarded((Tq, H, d), torch.bfloat16)
    lflat, lse = guarded_lse(H, Tq)
    fa.fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, max_q, max_k, scale, causal)
    fa.fa_device_status()
    o_in = torch.nan_to_num(o, nan=0.0)  # rows of broken sequences may stay unwritten
    lse_in = torch.nan_to_num(lse, nan=0.0)
    bufs = [guarded((Tq, H, d), torch.bfloat16), guarded((Tk, Hkv, d), torch.bfloat16),
            guarded((Tk, Hkv, d), torch.bfloat16)]
    ws = torch.empty(fa.fa_bwd_varlen_workspace_bytes(Tq, H, d), dtype=torch.uint8, device="cuda")
    fa.fa_bwd_varlen(q, k, v, o_in, do, lse_in, bufs[0][1], bufs[1][1], bufs[2][1], cu_q, cu_k,
                     max_q, max_k, scale, causal, ws)
    fa.fa_device_status()
    out = {"o": o.clone(), "lse": lse.clone(), "dq": bufs[0][1].clone(), "dk": bufs[1][1].clone(),
           "dv": bufs[2][1].clone()}
    assert_guards_intact(obuf, "o")
    assert_flat_guards_intact(lflat, "lse")
    for name, (b, _) in zip(("dq", "dk", "dv"), bufs):
        assert_guards_intact(b, name)
    if max_q <= 128:
        dbuf, od = guarded((Tq, H, d), torch.bfloat16)
        dflat, lsed = guarded_lse(H, Tq)
        need = fa.fa_decode_workspace_bytes(Tq, H, d, splits)
        wbuf = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
        fa.fa_fwd_decode(q, k, v, od, lsed, cu_q, cu_k, max_q, max_k, scale, causal, splits,
                         wbuf if need else None)
        fa.fa_device_status()
        assert_guards_intact(dbuf, "decode o")
        assert_flat_guards_intact(dflat, "decode lse")
        assert (wbuf[need:] == 0xA5).all(), "write past the decode workspace"
        out["od"], out["lsed"] = od.clone(), lsed.clone()
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_checked_matches_regular_bit_for_bit(checked, causal):
    lens_q, lens_k = [100, 0, 1, 128], [300, 5, 0, 129]
    x = random_varlen(lens_q, lens_k, 4, 2, 64, seed=11 + causal)
    cu_q, cu_k = x["cu_q"].cuda(), x["cu_k"].cuda()
    got = run_packed(x, cu_q, cu_k, 128, 300, causal, splits=3)
    with _lib.library(_lib.LIB_PATH):
        assert not fa.fa_checked_build()
        ref = run_packed(x, cu_q, cu_k, 128, 300, causal, splits=3)
    for name in ref:
        assert torch.equal(torch.nan_to_num(got[name]), torch.nan_to_num(ref[name])), name
    # fixed-length calls, including the fp32 path
    for dtype in (torch.bfloat16, torch.float32):
        y = random_qkv(2, 3, 200, 128, dtype=dtype, seed=4)
        q, k, v, do = (y[n].cuda() for n in ("q", "k", "v", "do"))
        res = []
        for path in (_lib.LIB_CHECKED_PATH, _lib.LIB_PATH):
            with _lib.library(path):
                o, lse = fa.forward(q, k, v, causal=causal)
                res.append((o, lse, *fa.backward(q, k, v, o, do, lse, causal=causal)))
                fa.fa_device_status()
        for a, b in zip(*res):
            assert torch.equal(a, b)
    # the e4m3 forward
    from exact_attention_25_gb300.inputs import random_fp8

    z = random_fp8(2, 2, 300, 128, seed=6)
    q8, k8, v8 = (z[n].cuda() for n in ("q", "k", "v"))
    res = []
    for path in (_lib.LIB_CHECKED_PATH, _lib.LIB_PATH):
        with _lib.library(path):
            res.append(fa.forward_fp8(q8, k8, v8, z["q_descale"], z["k_descale"], z["v_descale"],
                                      causal=causal))
            fa.fa_device_status()
    for a, b in zip(*res):
        assert torch.equal(a, b)


# (lens of the tensors, cu_q, cu_k, max_q, max_k): malformed offsets of several kinds
MALFORMED = [
    ("not monotonic", 400, 400, [0, 300, 100, 400], [0, 250, 50, 400], 128, 300),
    ("past the end", 400, 500, [0, 100, 5000], [0, 200, 900], 128, 400),
    ("negative", 300, 300, [-50, 100, 300], [-1000, 150, 300], 128, 300),
    ("longer than max", 400, 600, [0, 400], [0, 600], 64, 128),
    ("all beyond", 64, 64, [70, 80, 90], [100, 100, 200], 16, 64),
    ("decreasing to negative", 200, 200, [0, 200, -5, 100], [0, 200, 100, -300], 128, 200),
]


@pytest.mark.parametrize("case", MALFORMED, ids=[c[0] for c in MALFORMED])
@pytest.mark.parametrize("causal", [False, True])
def test_malformed_offsets_stay_inside_the_buffers(checked, case, causal):
    _, Tq, Tk, cq, ck, max_q, max_k = case
    B = len(cq) - 1
    # packed tensors of Tq query and Tk key rows, addressed through the malformed offsets
    x = random_varlen([Tq] + [0] * (B - 1), [Tk] + [0] * (B - 1), 4, 2, 128, seed=Tq + Tk)
    cu_q = torch.tensor(cq, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(ck, dtype=torch.int32, device="cuda")
    for splits in (1, 3):
        run_packed(x, cu_q, cu_k, max_q, max_k, causal, splits)


@pytest.mark.parametrize("case", MALFORMED, ids=[c[0] for c in MALFORMED])
def test_malformed_offsets_e4m3_stay_inside_the_buffers(checked, case):
    """The packed e4m3 forward (its V transpose reads through the same clamped offsets)."""
    from exact_attention_25_gb300.inputs import random_fp8_varlen

    _, Tq, Tk, cq, ck, max_q, max_k = case
    B = len(cq) - 1
    x = random_fp8_varlen([Tq] + [0] * (B - 1), [Tk] + [0] * (B - 1), 4, 2, 128, seed=Tq)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    cu_q = torch.tensor(cq, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(ck, dtype=torch.int32, device="cuda")
    obuf, o = guarded((Tq, 4, 128), torch.bfloat16)
    lflat, lse = guarded_lse(4, Tq)
    need = fa.fa_fwd_fp8_varlen_workspace_bytes(B, max_k, 2, 128)
    wbuf = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    for causal in (False, True):
        fa.fa_fwd_fp8_varlen(q, k, v, o, lse, cu_q, cu_k, max_q, max_k, 0.1, 1.0, 1.0, 1.0,
                             causal, wbuf)
        fa.fa_device_status()
    assert_guards_intact(obuf, "o")
    assert_flat_guards_intact(lflat, "lse")
    assert (wbuf[need:] == 0xA5).all(), "write past the workspace"


def expect_out_of_bounds(call):
    call()
    with pytest.raises(fa.FaError) as ei:
        fa.fa_device_status()
    assert ei.value.code == -9


def test_shrunk_extents_are_caught(checked):
    """Every extent one row step short: the call reports FA_ERR_OUT_OF_BOUNDS and the
    accesses past the shortened extent are skipped."""
    x = random_varlen([90, 200], [150, 200], 4, 2, 64, seed=3)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    cu_q, cu_k = x["cu_q"].cuda(), x["cu_k"].cuda()
    o_ref, lse_ref = fa.forward_varlen(q, k, v, cu_q, cu_k, 200, 200, causal=True)
    fa.fa_device_status()
    checked.fa_debug_set_flags(SHRINK_EXTENTS)
    try:
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        expect_out_of_bounds(lambda: fa.fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, 200, 200,
                                                      0.125, True))
        # O loses its last token row (one row step = H*d elements), lse its last element
        assert torch.isnan(o[-1].float()).all() and torch.isnan(lse[-1, -1])
        assert torch.equal(lse[-1, :-1], lse_ref[-1, :-1])
        assert torch.equal(o[:-1], o_ref[:-1]) and torch.equal(lse[:-1], lse_ref[:-1])
        grads = [torch.empty_like(t) for t in (q, k, v)]
        ws = torch.empty(fa.fa_bwd_varlen_workspace_bytes(q.shape[0], 4, 64), dtype=torch.uint8,
                         device="cuda")
        expect_out_of_bounds(lambda: fa.fa_bwd_varlen(q, k, v, o_ref, do, lse_ref, *grads, cu_q,
                                                      cu_k, 200, 200, 0.125, True, ws))
        for splits in (1, 2):
            need = fa.fa_decode_workspace_bytes(q.shape[0], 4, 64, splits)
            wsd = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
            y = random_varlen([3, 5], [150, 200], 4, 2, 64, seed=5)
            qd, kd, vd = (y[n].cuda() for n in ("q", "k", "v"))
            od = torch.empty_like(qd)
            lsed = torch.empty((4, qd.shape[0]), dtype=torch.float32, device="cuda")
            expect_out_of_bounds(lambda: fa.fa_fwd_decode(
                qd, kd, vd, od, lsed, y["cu_q"].cuda(), y["cu_k"].cuda(), 5, 200, 0.125, True,
                splits, wsd if need else None))
        # fixed-length forward and backward
        z = random_qkv(1, 2, 130, 128, seed=9)
        qf, kf, vf, dof = (z[n].cuda() for n in ("q", "k", "v", "do"))
        of, lsef = torch.empty_like(qf), torch.empty((1, 2, 130), dtype=torch.float32,
                                                     device="cuda")
        expect_out_of_bounds(lambda: fa.fa_fwd(qf, kf, vf, of, lsef, 0.1, False))
    finally:
        checked.fa_debug_set_flags(0)
    # back to normal: no report
    fa.forward_varlen(q, k, v, cu_q, cu_k, 200, 200, causal=True)
    fa.fa_device_status()


def test_shrunk_extents_are_caught_in_the_fixed_length_backward(checked):
    """The same hook on the fixed-length bf16 backward (the preprocess, the dK/dV kernel's
    stores and the dQ kernel's stores are all checked); with the hook off again the call
    reports nothing."""
    z = random_qkv(1, 2, 130, 128, seed=9)
    q, k, v, do = (z[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True)
    fa.fa_device_status()
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, 2, 130, 128), dtype=torch.uint8, device="cuda")
    grads = [torch.empty_like(t) for t in (q, k, v)]
    checked.fa_debug_set_flags(SHRINK_EXTENTS)
    try:
        expect_out_of_bounds(lambda: fa.fa_bwd(q, k, v, o, do, lse, *grads, 0.1, True, ws))
    finally:
        checked.fa_debug_set_flags(0)
    fa.fa_bwd(q, k, v, o, do, lse, *grads, 0.1, True, ws)
    fa.fa_device_status()
