"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory (it keeps its
scratch in a fixed array inside the library instead of a caller workspace).  Checked through
the C ABI against fa_bwd on the same inputs, on two calls in a row.  This file is collected
last so that a run stopping at the first failure has already run every other test."""
import ctypes

import pytest
import torch

import exact_attention_25_gb300 as fa
from exact_attention_25_gb300.inputs import random_qkv
from tests.gpu_util import TOL_GRAD_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, scale, causal):
    B, H, N, d = q.shape
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.fa_bwd_noalloc(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), B, H, N,
                              d, ctypes.c_float(scale), int(causal), fa.FA_BF16,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_backward_matches_fa_bwd_on_two_calls(causal):
    lib = fa.load()
    B, H, N, d = 1, 3, 777, 128
    x = random_qkv(B, H, N, d, seed=4242)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    ref = fa.backward(q, k, v, o, do, lse, scale=scale, causal=causal)
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        rc = _noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, scale, causal)
        assert rc == 0, (rc, lib.fa_last_error().decode())
        fa.fa_device_status()
        for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            assert torch.isfinite(got.float()).all(), (call, name)
            assert rel_l2(got, want) <= TOL_GRAD_REL_L2, (call, name, rel_l2(got, want))


def test_noalloc_rejects_shapes_beyond_its_array():
    lib = fa.load()
    A = ctypes.c_void_p(0x10000)
    rc = lib.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, 1, 32, 40000, 128, ctypes.c_float(0.1), 1,
                            fa.FA_BF16, None)
    assert rc == -7 and "1048576" in lib.fa_last_error().decode()
