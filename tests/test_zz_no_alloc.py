"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory (it keeps its
scratch in a fixed array inside the library instead of a caller workspace).  Checked through
the C ABI against fa_bwd on the same inputs: both run the same deterministic kernels, so the
gradients must be equal bit for bit.  The two calls in a row differ in seed, shape and mask,
so a call that read scratch left behind by the one before would show.  One case uses exactly
the largest accepted size (B*H*N = 2^20 rows, the whole array), also through the checked
build, whose kernels test every access against its buffer.  This file is collected last so
that a run stopping at the first failure has already run every other test."""
import ctypes

import pytest
import torch

import exact_attention_25_gb300 as fa
from exact_attention_25_gb300 import _lib
from exact_attention_25_gb300.inputs import random_qkv

pytestmark = pytest.mark.gpu

MAX_ROWS = 1 << 20


def _noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, scale, causal):
    B, H, N, d = q.shape
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dtype = fa.FA_F32 if q.dtype == torch.float32 else fa.FA_BF16
    return lib.fa_bwd_noalloc(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), B, H, N,
                              d, ctypes.c_float(scale), int(causal), dtype,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _compare_with_fa_bwd(lib, B, H, N, d, causal, seed, dtype=torch.bfloat16):
    """One fa_bwd_noalloc call on fresh inputs; its gradients must equal fa_bwd's bit for bit."""
    x = random_qkv(B, H, N, d, dtype=dtype, seed=seed)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = d ** -0.5
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    ref = fa.backward(q, k, v, o, do, lse, scale=scale, causal=causal)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    rc = _noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, scale, causal)
    assert rc == 0, (rc, lib.fa_last_error().decode())
    rc = lib.fa_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, (rc, lib.fa_last_error().decode())
    for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        assert torch.equal(got, want), (B, H, N, d, causal, name,
                                        float((got.float() - want.float()).abs().max()))


def test_noalloc_two_calls_in_a_row_equal_fa_bwd():
    lib = fa.load()
    _compare_with_fa_bwd(lib, 1, 3, 777, 128, False, seed=4242)
    _compare_with_fa_bwd(lib, 2, 2, 1000, 64, True, seed=4243)


def test_noalloc_fp32_path_equals_fa_bwd():
    lib = fa.load()
    _compare_with_fa_bwd(lib, 1, 2, 300, 64, True, seed=4244, dtype=torch.float32)
    _compare_with_fa_bwd(lib, 2, 1, 129, 128, False, seed=4245, dtype=torch.float32)


def test_noalloc_at_the_largest_accepted_size():
    """B*H*N = 2^20 rows: the scratch for the base-2 LSE ends on the last byte of the array."""
    B, H, N, d = 2, 128, 4096, 64
    assert B * H * N == MAX_ROWS
    _compare_with_fa_bwd(fa.load(), B, H, N, d, True, seed=4246)


def test_noalloc_at_the_largest_accepted_size_checked_build():
    """The same size through libfa_checked.so: every direct global access of the kernels is
    tested against its buffer's extent, so an access past the array or the outputs would be
    reported by fa_device_status as FA_ERR_OUT_OF_BOUNDS."""
    B, H, N, d = 2, 128, 4096, 64
    with _lib.library(_lib.LIB_CHECKED_PATH) as lib:
        assert lib.fa_checked_build() == 1
        _compare_with_fa_bwd(lib, B, H, N, d, True, seed=4247)


def test_noalloc_rejects_shapes_beyond_its_array():
    lib = fa.load()
    A = ctypes.c_void_p(0x10000)
    rc = lib.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, 1, 32, 40000, 128, ctypes.c_float(0.1), 1,
                            fa.FA_BF16, None)
    assert rc == -7 and "1048576" in lib.fa_last_error().decode()
    # one row more than the array holds
    rc = lib.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, 1, 1, MAX_ROWS + 1, 64, ctypes.c_float(0.1),
                            1, fa.FA_BF16, None)
    assert rc == -7
