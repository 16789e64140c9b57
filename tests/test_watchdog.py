"""Bounded device waits: a wait that can never complete expires after the configured limit,
the kernel returns without faulting or hanging, fa_device_status() reports the timeout, and
the CUDA context stays usable.  The failure is made by a test hook that announces a tile but
never copies it (no invalid memory access, no trap)."""
import pytest
import torch

import exact_attention_25_gb300 as fa
from exact_attention_25_gb300 import _lib
from exact_attention_25_gb300.inputs import random_qkv, random_varlen

pytestmark = pytest.mark.gpu


@pytest.fixture
def short_waits():
    lib = fa.load()
    fa.fa_set_wait_limit_ns(20_000_000)  # 20 ms
    yield lib
    lib.fa_debug_set_flags(0)
    fa.fa_set_wait_limit_ns(2_000_000_000)


def _expect_timeout():
    with pytest.raises(fa.FaError) as ei:
        fa.fa_device_status()
    assert ei.value.code == -6, ei.value
    assert "site" in _lib.last_error()


def test_forward_wait_expires_and_context_survives(short_waits):
    x = random_qkv(1, 1, 200, 128, seed=1, with_do=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    short_waits.fa_debug_set_flags(1)
    fa.forward(q, k, v, causal=True)
    _expect_timeout()
    short_waits.fa_debug_set_flags(0)
    o, lse = fa.forward(q, k, v, causal=True)
    fa.fa_device_status()  # clean again
    assert torch.isfinite(o.float()).all()


def test_backward_wait_expires_and_context_survives(short_waits):
    x = random_qkv(1, 1, 200, 128, seed=2)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=False)
    fa.fa_device_status()
    short_waits.fa_debug_set_flags(1)
    fa.backward(q, k, v, o, do, lse, causal=False)
    _expect_timeout()
    short_waits.fa_debug_set_flags(0)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=False)
    fa.fa_device_status()
    assert torch.isfinite(dq.float()).all() and torch.isfinite(dv.float()).all()


def test_decode_wait_expires_and_context_survives(short_waits):
    x = random_varlen([1, 1], [300, 500], 8, 2, 128, seed=3, with_do=False)
    q, k, v, cu_q, cu_k = (x[n].cuda() for n in ("q", "k", "v", "cu_q", "cu_k"))
    short_waits.fa_debug_set_flags(1)
    fa.forward_decode(q, k, v, cu_q, cu_k, 1, 500, causal=True, num_splits=2)
    _expect_timeout()
    short_waits.fa_debug_set_flags(0)
    o, lse = fa.forward_decode(q, k, v, cu_q, cu_k, 1, 500, causal=True, num_splits=2)
    fa.fa_device_status()
    assert torch.isfinite(o.float()).all()


def test_fp8_forward_wait_expires_and_context_survives(short_waits):
    from exact_attention_25_gb300.inputs import random_fp8

    x = random_fp8(1, 2, 600, 128, seed=4)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    short_waits.fa_debug_set_flags(1)
    fa.forward_fp8(q, k, v, causal=True)
    _expect_timeout()
    short_waits.fa_debug_set_flags(0)
    o, lse = fa.forward_fp8(q, k, v, causal=True)
    fa.fa_device_status()
    assert torch.isfinite(o.float()).all()
