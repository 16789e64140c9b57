"""Host-side checks of the C ABI that need no GPU: the library loads, exports every symbol the
header declares, rejects bad arguments with the documented codes before touching CUDA, and
its causal block schedule matches the counts printed in the Triton FA2 write-up."""
import ctypes
import json
import math
import os
import re

import pytest

from exact_attention_25_gb300 import _lib, build, perfmodel


def _no_device():
    import torch

    return not torch.cuda.is_available()


# A call with dummy pointers that passes every host check goes on to launch.  Such calls are made
# only where no CUDA device exists (the call then fails at the device query); with a device they
# would launch kernels on addresses that are not allocations.
LAUNCH_SAFE = _no_device()

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load(_lib.LIB_PATH)  # the regular library, whatever FA_CHECKED says


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_expected_entry_points():
    names = declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_device_status"} <= set(names)
    assert set(names) == set(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_checked_variant_exports_the_same_symbols_and_says_so(lib):
    path = build.build(checked=True)
    checked = _lib.load(path)
    for name in declared_functions():
        assert hasattr(checked, name), name
    assert checked.fa_checked_build() == 1 and lib.fa_checked_build() == 0
    # argument validation is shared: the checked variant rejects the same calls
    assert fwd(checked, d=96) == -2 and fwd(checked, q=MIS) == -3


P = ctypes.c_void_p
A = P(0x10000)  # aligned dummy pointers: validation must reject before dereferencing
A2 = P(0x20000)
MIS = P(0x10008)


def fwd(lib, q=A, k=A, v=A, o=A2, lse=A2, B=1, H=1, N=8, d=64, scale=0.125, causal=0, dtype=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), causal, dtype, None)


def fp8(lib, q=A, k=A, v=A, o=A2, lse=A2, B=1, H=1, N=8, d=128, scale=0.1, qd=1.0, kd=1.0,
        vd=1.0, causal=0, ws=A, nbytes=1 << 20):
    f = ctypes.c_float
    return lib.fa_fwd_fp8(q, k, v, o, lse, B, H, N, d, f(scale), f(qd), f(kd), f(vd), causal, ws,
                          nbytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), -2), (dict(N=0), -1), (dict(q=None), -1), (dict(ws=None), -4),
    (dict(nbytes=16), -4), (dict(qd=math.inf), -1), (dict(vd=math.nan), -1),
    (dict(scale=1e30, qd=1e30), -1), (dict(k=MIS), -3), (dict(ws=MIS), -3), (dict(causal=3), -1),
])
def test_fp8_forward_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert fp8(lib, **kw) == code


def fp8_varlen(lib, cu_q=A, cu_k=A, B=2, max_q=64, max_k=64, total_q=100, total_k=100, H=4,
               Hkv=2, d=128, ws=A, nbytes=1 << 24, qd=1.0):
    f = ctypes.c_float
    return lib.fa_fwd_fp8_varlen(A, A, A, A2, A2, cu_q, cu_k, B, max_q, max_k, total_q, total_k,
                                 H, Hkv, d, f(0.1), f(qd), f(1.0), f(1.0), 0, ws, nbytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), -2), (dict(B=0), -1), (dict(cu_q=None), -1), (dict(H=3), -1),
    (dict(ws=None), -4), (dict(nbytes=256), -4), (dict(qd=math.inf), -1), (dict(ws=MIS), -3),
])
def test_fp8_varlen_forward_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert fp8_varlen(lib, **kw) == code


def test_fp8_varlen_workspace_size_contract(lib):
    # V^T per (sequence, key/value head), keys padded to 16
    assert lib.fa_fwd_fp8_varlen_workspace_bytes(3, 100, 2, 128) >= 3 * 2 * 128 * 112
    assert lib.fa_fwd_fp8_varlen_workspace_bytes(0, 100, 2, 128) == 0


def test_fp8_workspace_size_contract(lib):
    # one transposed copy of V, keys padded to a multiple of 16
    assert lib.fa_fwd_fp8_workspace_bytes(2, 3, 100, 128) >= 2 * 3 * 128 * 112
    assert lib.fa_fwd_fp8_workspace_bytes(1, 1, 16, 128) >= 128 * 16
    assert lib.fa_fwd_fp8_workspace_bytes(0, 1, 16, 128) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), -2), (dict(d=32), -2), (dict(N=0), -1), (dict(B=0), -1), (dict(H=-1), -1),
    (dict(q=None), -1), (dict(o=None), -1), (dict(dtype=5), -1), (dict(causal=2), -1),
    (dict(scale=math.inf), -1), (dict(scale=math.nan), -1), (dict(q=MIS), -3), (dict(o=MIS), -3),
    (dict(B=1024, H=1024, N=1024, d=128), -7),
])
def test_forward_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert fwd(lib, **kw) == code
    assert lib.fa_last_error().decode() != ""


def bwd(lib, ws=A, ws_bytes=None, **kw):
    args = dict(B=1, H=2, N=100, d=128, scale=0.1, causal=1, dtype=0)
    args.update(kw)
    if ws_bytes is None:
        ws_bytes = lib.fa_bwd_workspace_bytes(args["B"], args["H"], args["N"], args["d"])
    return lib.fa_bwd(A, A, A, A, A, A, A2, A2, A2, args["B"], args["H"], args["N"], args["d"],
                      ctypes.c_float(args["scale"]), args["causal"], args["dtype"], ws, ws_bytes,
                      None)


def test_backward_rejects_bad_arguments(lib):
    assert bwd(lib, d=80) == -2
    assert bwd(lib, N=0) == -1
    assert bwd(lib, ws=None) == -4
    need = lib.fa_bwd_workspace_bytes(1, 2, 100, 128)
    assert need >= 2 * 200 * 4
    assert bwd(lib, ws_bytes=need - 1) == -4
    assert bwd(lib, ws=MIS) == -3


def test_backward_rejects_outputs_that_overlap_another_tensor(lib):
    # B1 H2 N100 d128 bf16: 51200 bytes per tensor; tensors 1 MiB apart do not touch
    B, H, N, d = 1, 2, 100, 128
    need = lib.fa_bwd_workspace_bytes(B, H, N, d)
    base = 0x1000000
    names = ["q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv", "ws"]
    addr = {n: base + i * (1 << 20) for i, n in enumerate(names)}

    def call(**place):  # place: tensor -> (other tensor, byte offset from its start)
        a = dict(addr)
        for n, (other, off) in place.items():
            a[n] = addr[other] + off
        a = {n: P(x) for n, x in a.items()}
        return lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"],
                          a["dv"], B, H, N, d, ctypes.c_float(0.1), 1, 0, a["ws"], need, None)

    # disjoint tensors pass validation (no GPU here: the call then fails with another code)
    if LAUNCH_SAFE:  # passes the host checks
        assert call() != -1
    # dq over the end of q, dk over dq's last 16 bytes, dv inside the workspace, dk on lse
    assert call(dq=("q", 51200 - 16)) == -1
    assert "overlap" in lib.fa_last_error().decode()
    assert call(dk=("dq", 51200 - 16)) == -1
    assert call(dv=("ws", need - 16)) == -1
    assert call(dk=("lse", 800 - 16)) == -1
    # a tensor that ends exactly where the next begins does not overlap it
    if LAUNCH_SAFE:  # passes the host checks
        assert call(dq=("q", 51200)) != -1
    if LAUNCH_SAFE:  # passes the host checks
        assert call(dk=("lse", 800)) != -1

    def gqa(dq_at):
        ws = lib.fa_bwd_workspace_bytes(1, 4, 10, 128)
        return lib.fa_bwd_gqa(P(0x1000000), P(0x2000000), P(0x3000000), P(0x4000000),
                              P(0x5000000), P(0x6000000), P(dq_at), P(0x8000000), P(0x9000000),
                              1, 4, 2, 10, 20, 128, ctypes.c_float(0.1), 1, P(0xA000000), ws,
                              None)

    if LAUNCH_SAFE:  # passes the host checks
        assert gqa(0x7000000) != -1
    assert gqa(0x5000000 + 4 * 10 * 128 * 2 - 16) == -1  # dq over the end of dout


def test_workspace_size_contract(lib):
    assert lib.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0
    assert lib.fa_bwd_workspace_bytes(1, 1, 1, 96) == 0
    for (B, H, N) in [(1, 1, 1), (4, 16, 4096), (1, 32, 32000)]:
        assert lib.fa_bwd_workspace_bytes(B, H, N, 128) >= 2 * B * H * N * 4


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.fa_status_string(code).decode() == name
    assert lib.fa_version().decode().startswith("fa-gb300")


def counts(lib, q_block, Br, Bc, N):
    nf, nm = ctypes.c_int(), ctypes.c_int()
    rc = lib.fa_causal_block_counts(q_block, Br, Bc, N, ctypes.byref(nf), ctypes.byref(nm))
    assert rc == 0
    return nf.value, nm.value


def test_causal_schedule_matches_the_printed_counts(lib):
    g = json.load(open(os.path.join(GOLDEN, "causal_blocks.json")))
    for c in g["cases"]:
        assert counts(lib, c["q_block"], c["Br"], c["Bc"], c["N"]) == (c["n_full"], c["n_masked"]), c


@pytest.mark.parametrize("Br,Bc,N", [(128, 128, 1000), (64, 128, 777), (128, 64, 4096), (256, 128, 2000),
                                     (128, 128, 1), (7, 5, 100)])
def test_causal_schedule_against_brute_force(lib, Br, Bc, N):
    """Block classes against a per-element scan of the key <= query mask."""
    for qb in range((N + Br - 1) // Br):
        q0, q1 = qb * Br, min(N, (qb + 1) * Br)
        nf = nm = 0
        for k0 in range(0, N, Bc):
            k1 = min(N, k0 + Bc)
            vis = [[j <= i for j in range(k0, k1)] for i in range(q0, q1)]
            flat = [x for r in vis for x in r]
            if all(flat):
                nf += 1
            elif any(flat):
                nm += 1
        assert counts(lib, qb, Br, Bc, N) == (nf, nm), (qb, Br, Bc, N)
    assert lib.fa_causal_block_counts((N + Br - 1) // Br, Br, Bc, N, ctypes.byref(ctypes.c_int()),
                                      ctypes.byref(ctypes.c_int())) == -1


def test_hbm_models_match_the_printed_tables():
    g = json.load(open(os.path.join(GOLDEN, "hbm_models.json")))
    sa = g["standard_attention_fp16"]
    for N, b in sa["rows"]:
        assert abs(perfmodel.standard_attention_intermediate_bytes(N, 2) - b) <= sa["rel_tol"] * b
    l6 = g["lesson06_fp32_d64"]
    for N, naive_mib, flash_mib in l6["rows"]:
        naive, flash = perfmodel.lesson06_hbm_elements(N, l6["d"])
        assert abs(naive * 4 / 2**20 - naive_mib) <= l6["rel_tol"] * naive_mib + 0.05
        assert abs(flash * 4 / 2**20 - flash_mib) <= l6["rel_tol"] * flash_mib
    t = g["tiling_example"]
    assert t["Br"] * t["d"] * t["elem_bytes"] == t["tile_kb"] * 1024
    assert 5 * t["tile_kb"] == t["total_kb"]
    assert math.ceil(t["N"] / t["Br"]) == t["Tr"] and math.ceil(t["N"] / t["Bc"]) == t["Tc"]


def test_flop_convention():
    assert perfmodel.fwd_flops(1, 1, 512, 64, False) == 4 * 512 * 512 * 64
    assert perfmodel.fwd_flops(2, 32, 8192, 128, True) == pytest.approx(1.0995e12, rel=1e-4)
    assert perfmodel.bwd_flops(4, 16, 4096, 128, True) == pytest.approx(6.872e11, rel=1e-3)


def fwd_varlen(lib, cu_q=A, cu_k=A, B=2, max_q=10, max_k=10, total_q=20, total_k=20, H=4, Hkv=2,
               d=128, scale=0.1, causal=1, q=A, o=A2):
    return lib.fa_fwd_varlen(q, A, A, o, A2, cu_q, cu_k, B, max_q, max_k, total_q, total_k, H,
                             Hkv, d, ctypes.c_float(scale), causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(H=4, Hkv=3), -1), (dict(Hkv=0), -1), (dict(B=0), -1), (dict(total_q=0), -1),
    (dict(max_k=0), -1), (dict(d=96), -2), (dict(cu_q=None), -1), (dict(cu_k=None), -1),
    (dict(cu_q=P(0x10002)), -3), (dict(q=MIS), -3), (dict(causal=3), -1),
    (dict(scale=math.nan), -1), (dict(total_q=1 << 20, H=64, d=128), -7),
])
def test_varlen_forward_rejects_bad_arguments_before_any_launch(lib, kw, code):
    assert fwd_varlen(lib, **kw) == code
    assert lib.fa_last_error().decode() != ""


def test_varlen_backward_rejects_bad_arguments(lib):
    need = lib.fa_bwd_varlen_workspace_bytes(20, 4, 128)
    assert need >= 2 * 20 * 4 * 4
    assert lib.fa_bwd_varlen_workspace_bytes(0, 4, 128) == 0
    assert lib.fa_bwd_varlen_workspace_bytes(20, 4, 80) == 0

    def call(ws=A, nbytes=need, H=4, Hkv=2):
        return lib.fa_bwd_varlen(A, A, A, A, A, A, A2, A2, A2, A, A, 2, 10, 10, 20, 20, H, Hkv,
                                 128, ctypes.c_float(0.1), 1, ws, nbytes, None)

    assert call(ws=None) == -4
    assert call(nbytes=need - 1) == -4
    assert call(ws=MIS) == -3
    assert call(H=5) == -1


def test_varlen_backward_rejects_overlapping_outputs_unless_strided(lib):
    # 20 query and 20 key tokens, H4 over Hkv2, d128 bf16: q-side tensors 20480 bytes,
    # k-side 10240, lse 320; tensors 1 MiB apart do not touch
    need = lib.fa_bwd_varlen_workspace_bytes(20, 4, 128)
    names = ["q", "k", "v", "o", "do", "lse", "dq", "dk", "dv", "ws"]
    addr = {n: 0x1000000 + i * (1 << 20) for i, n in enumerate(names)}

    def call(strides=None, **place):
        a = dict(addr)
        for n, (other, off) in place.items():
            a[n] = addr[other] + off
        a = {n: P(x) for n, x in a.items()}
        args = [a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"]]
        tail = [A, A, 2, 10, 10, 20, 20, 4, 2, 128, ctypes.c_float(0.1), 1, a["ws"], need, None]
        if strides is None:
            return lib.fa_bwd_varlen(*args, *tail)
        return lib.fa_bwd_varlen_strided(*args, strides, *tail)

    if LAUNCH_SAFE:  # passes the host checks
        assert call() != -1
    assert call(dq=("do", 20480 - 16)) == -1
    assert "overlap" in lib.fa_last_error().decode()
    assert call(dv=("dk", 10240 - 16)) == -1
    assert call(dk=("ws", 0)) == -1
    if LAUNCH_SAFE:  # passes the host checks
        assert call(dq=("do", 20480)) != -1
    # strided views may interleave in one buffer: not checked
    arr = (ctypes.c_longlong * 16)(*([512, 128] * 4 + [512, 128] + [512, 128] + [256, 128] * 2))
    if LAUNCH_SAFE:  # passes the host checks
        assert call(strides=arr, dq=("do", 20480 - 16)) != -1


def test_decode_rejects_bad_arguments(lib):
    need = lib.fa_decode_workspace_bytes(256, 32, 128, 4)
    assert need >= 4 * 256 * 32 * (128 + 1) * 4
    assert lib.fa_decode_workspace_bytes(8, 32, 128, 1) == 0
    assert lib.fa_decode_workspace_bytes(8, 32, 128, 0) == 0
    assert lib.fa_decode_workspace_bytes(8, 32, 96, 2) == 0

    def call(H=32, Hkv=8, max_q=1, splits=4, ws=A, nbytes=need, d=128):
        return lib.fa_fwd_decode(A, A, A, A2, A2, A, A, 8, max_q, 1000, 256, 8000, H, Hkv, d,
                                 ctypes.c_float(0.1), 1, splits, ws, nbytes, None)

    assert call(max_q=129) == -1           # more queries than one 128-row tile
    assert call(H=30) == -1                # H % Hkv
    assert call(splits=0) == -1
    assert call(splits=257) == -1
    assert call(ws=None) == -4
    assert call(nbytes=need - 1) == -4
    assert call(ws=MIS) == -3
    assert call(d=80) == -2
    assert lib.fa_decode_num_splits(0, 8, 100) == -1


def test_strided_varlen_rejects_bad_strides(lib):
    def fwd_st(vals):
        arr = None if vals is None else (ctypes.c_longlong * len(vals))(*vals)
        return lib.fa_fwd_varlen_strided(A, A, A, A2, A2, arr, A, A, 2, 10, 10, 20, 20, 4, 2, 128,
                                         ctypes.c_float(0.1), 1, None)

    good = [3 * 4 * 128, 128, 3 * 4 * 128, 128, 3 * 4 * 128, 128, 4 * 128, 128]
    assert fwd_st(None) == -1
    bad = list(good); bad[0] = 3 * 4 * 128 + 4          # row stride not a multiple of 8
    assert fwd_st(bad) == -3
    bad = list(good); bad[3] = 64                       # head step narrower than d = 128
    assert fwd_st(bad) == -1
    bad = list(good); bad[6] = 64; bad[7] = 128          # row step narrower than the head step
    assert fwd_st(bad) == -1
    bad = list(good); bad[5] = 0
    assert fwd_st(bad) == -3


def test_grouped_fixed_length_rejects_bad_arguments(lib):
    def call(B=1, H=4, Hkv=2, Nq=10, Nk=20, d=128, q=A):
        return lib.fa_fwd_gqa(q, A, A, A2, A2, B, H, Hkv, Nq, Nk, d, ctypes.c_float(0.1), 1, None)

    assert call(H=4, Hkv=3) == -1
    assert call(Nk=0) == -1
    assert call(d=96) == -2
    assert call(q=MIS) == -3
    assert call(B=1024, H=1024, Nq=1024, d=128) == -7

    def bcall(ws=A, nbytes=None):
        nb = lib.fa_bwd_workspace_bytes(1, 4, 10, 128) if nbytes is None else nbytes
        return lib.fa_bwd_gqa(A, A, A, A, A, A, A2, A2, A2, 1, 4, 2, 10, 20, 128,
                              ctypes.c_float(0.1), 1, ws, nb, None)

    assert bcall(ws=None) == -4
    assert bcall(nbytes=16) == -4


def test_decode_split_rule_takes_one_wave(lib):
    """The split count fa_decode_num_splits suggests (its host copy): the largest whose
    B * Hkv * splits CTAs all fit on the SMs at once, at least 8 key blocks of 128 per range."""
    f = lib.fa_decode_splits_for
    assert f(8, 8, 8192, 152) == 2      # 64 groups: 2 x 64 CTAs fit on 152 SMs, 3 x 64 do not
    assert f(8, 8, 32768, 152) == 2
    assert f(4, 8, 16384, 152) == 4
    assert f(2, 8, 32768, 152) == 9
    assert f(1, 8, 131072, 152) == 19
    assert f(16, 8, 8192, 152) == 1
    assert f(64, 8, 4096, 152) == 1     # more groups than SMs
    assert f(8, 8, 2048, 152) == 2      # 16 blocks: at most two ranges of 8
    assert f(1, 1, 1000, 152) == 1      # 8 blocks: one range
    assert f(1, 1, 10 ** 9, 152) == 152  # bounded by the SMs ...
    assert f(1, 1, 10 ** 9, 1000) == 256  # ... and by the 256-range limit
    for bad in [(0, 8, 100, 152), (8, 0, 100, 152), (8, 8, 0, 152), (8, 8, 100, 0)]:
        assert f(*bad) == -1


def _order(lib, id_, heads, nblk, gsize):
    h, r = ctypes.c_int(), ctypes.c_int()
    assert lib.fa_tile_order(id_, heads, nblk, gsize, ctypes.byref(h), ctypes.byref(r)) == 0
    return h.value, r.value


@pytest.mark.parametrize("heads,nblk,gsize", [(1, 1, 1), (64, 32, 16), (64, 32, 8), (7, 5, 3),
                                              (32, 250, 1), (5, 9, 16), (3, 4, 2)])
def test_tile_order_reaches_every_tile_once_heaviest_first_within_groups(lib, heads, nblk, gsize):
    """Every (head, rank) pair is reached by exactly one tile index; within a group of heads the
    ranks never decrease along the launch order (the heaviest tiles start first), the group's
    heads are interleaved, and groups follow one another."""
    seen = [_order(lib, i, heads, nblk, gsize) for i in range(heads * nblk)]
    assert sorted(seen) == [(h, r) for h in range(heads) for r in range(nblk)]
    for i, (h, r) in enumerate(seen):
        g0 = (h // gsize) * gsize
        gh = min(gsize, heads - g0)
        # the explicit position of (h, r): its group's start, then rank-major, head-minor
        assert i == g0 * nblk + r * gh + (h - g0), (i, h, r)
    if gsize == 1:  # head-major
        assert seen == [(h, r) for h in range(heads) for r in range(nblk)]


def test_tile_order_rejects_out_of_range_arguments(lib):
    h, r = ctypes.c_int(), ctypes.c_int()
    for args in ((-1, 2, 2, 1), (4, 2, 2, 1), (0, 0, 2, 1), (0, 2, 0, 1), (0, 2, 2, 0)):
        assert lib.fa_tile_order(*args, ctypes.byref(h), ctypes.byref(r)) == -1


def test_order_group_follows_the_l2_budget(lib):
    """Head-major without the causal mask; under it as many heads as keep 4 N d bytes each
    within 32 MB, between 1 and 16."""
    assert lib.fa_order_group(4096, 128, 0) == 1
    assert lib.fa_order_group(4096, 128, 1) == 16      # 2 MB per head
    assert lib.fa_order_group(8192, 128, 1) == 8       # 4 MB per head
    assert lib.fa_order_group(32000, 128, 1) == 2      # 16.4 MB per head
    assert lib.fa_order_group(131072, 128, 1) == 1     # 67 MB per head
    assert lib.fa_order_group(512, 64, 1) == 16
