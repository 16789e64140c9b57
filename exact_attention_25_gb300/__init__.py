"""GB300-native exact attention (FlashAttention-style forward and backward) for sm_103a.

The computation lives in ``libfa.so`` (hand-written CUDA: TMA, tcgen05/TMEM, warp-specialised
roles) behind the C ABI of ``include/fa.h``.  This module is the thin Python binding: the
``fa_*`` functions mirror the C entry points one to one and only marshal torch tensors into
pointers and sizes; ``forward``/``backward`` additionally allocate the outputs with torch.
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import FA_BF16, FA_F32, FaError, check, load

__all__ = [
    "FA_BF16", "FA_F32", "FaError", "load", "fa_fwd", "fa_bwd", "fa_bwd_stage", "fa_bwd_workspace_bytes",
    "fa_device_status", "fa_set_wait_limit_ns", "fa_causal_block_counts", "forward", "backward",
    "fa_fwd_varlen", "fa_bwd_varlen", "fa_bwd_varlen_workspace_bytes", "forward_varlen",
    "backward_varlen", "fa_fwd_decode", "fa_decode_workspace_bytes", "fa_decode_num_splits",
    "forward_decode", "fa_checked_build", "fa_fwd_fp8", "fa_fwd_fp8_workspace_bytes",
    "forward_fp8", "fa_fwd_fp8_varlen", "fa_fwd_fp8_varlen_workspace_bytes", "forward_fp8_varlen",
]


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:
        return FA_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _shape(q):
    if q.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    return tuple(int(x) for x in q.shape)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_tensors(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")


def _grouped(q, k) -> bool:
    """True when k has fewer heads or another length than q (the fa_*_gqa entry points)."""
    return tuple(k.shape[1:3]) != tuple(q.shape[1:3])


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool, stream=None, impl: int = 0) -> None:
    """C ``fa_fwd`` (``fa_fwd_impl`` when impl != 0): writes o and lse in place.  With k and v
    of shape [B, Hkv, Nk, d] other than q's [B, H, Nq, d] it calls ``fa_fwd_gqa``."""
    _check_tensors(q, k, v, o, lse)
    if _grouped(q, k):
        if impl:
            raise ValueError("grouped heads and Nq != Nk run on the tensor-core path only")
        B, H, Nq, d = _shape(q)
        _, Hkv, Nk, _ = _shape(k)
        check(load().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Nq, Nk,
                                d, float(scale), int(bool(causal)), _stream(stream)))
        return
    B, H, N, d = _shape(q)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
            int(bool(causal)), _dtype_code(q))
    lib = load()
    if impl:
        check(lib.fa_fwd_impl(*args, int(impl), _stream(stream)))
    else:
        check(lib.fa_fwd(*args, _stream(stream)))


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale: float, causal: bool, workspace,
           stream=None, impl: int = 0) -> None:
    """C ``fa_bwd`` (``fa_bwd_impl`` when impl != 0): writes dq, dk, dv in place; grouped or
    non-square shapes call ``fa_bwd_gqa``."""
    _check_tensors(q, k, v, o, do, lse, dq, dk, dv, workspace)
    nbytes = workspace.numel() * workspace.element_size()
    if _grouped(q, k):
        if impl:
            raise ValueError("grouped heads and Nq != Nk run on the tensor-core path only")
        B, H, Nq, d = _shape(q)
        _, Hkv, Nk, _ = _shape(k)
        check(load().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                _ptr(dk), _ptr(dv), B, H, Hkv, Nq, Nk, d, float(scale),
                                int(bool(causal)), _ptr(workspace), nbytes, _stream(stream)))
        return
    B, H, N, d = _shape(q)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv), B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q), _ptr(workspace),
            nbytes)
    lib = load()
    if impl:
        check(lib.fa_bwd_impl(*args, int(impl), _stream(stream)))
    else:
        check(lib.fa_bwd(*args, _stream(stream)))


def fa_bwd_stage(q, k, v, o, do, lse, dq, dk, dv, scale: float, causal: bool, workspace,
                 stage: int, stream=None) -> None:
    """C ``fa_bwd_stage``: 0 = preprocess, 1 = dK/dV, 2 = dQ (0, 1, 2 in order = fa_bwd)."""
    _check_tensors(q, k, v, o, do, lse, dq, dk, dv, workspace)
    B, H, N, d = _shape(q)
    nbytes = workspace.numel() * workspace.element_size()
    check(load().fa_bwd_stage(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q), _ptr(workspace), nbytes,
        int(stage), _stream(stream)))


def fa_device_status(stream=None) -> None:
    """C ``fa_device_status``: synchronises and raises FaError if a device wait timed out."""
    check(load().fa_device_status(_stream(stream)))


def fa_set_wait_limit_ns(ns: int) -> None:
    load().fa_set_wait_limit_ns(int(ns))


def fa_checked_build() -> bool:
    """C ``fa_checked_build``: whether the library in use is the bounds-checked variant."""
    return bool(load().fa_checked_build())


def fa_fwd_fp8_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_fwd_fp8_workspace_bytes(B, H, N, d))


def fa_fwd_fp8(q, k, v, o, lse, scale: float, q_descale: float, k_descale: float,
               v_descale: float, causal: bool, workspace, stream=None) -> None:
    """C ``fa_fwd_fp8``: q, k, v [B, H, N, 128] e4m3 codes (any 1-byte dtype, for example
    torch.float8_e4m3fn or uint8), o [B, H, N, 128] bf16, lse [B, H, N] fp32 or None."""
    _check_tensors(q, k, v, o, lse, workspace)
    for t in (q, k, v):
        if t.element_size() != 1 or tuple(t.shape) != tuple(q.shape):
            raise ValueError("q, k and v must be [B, H, N, d] tensors of 1-byte e4m3 codes")
    B, H, N, d = _shape(q)
    nbytes = workspace.numel() * workspace.element_size()
    check(load().fa_fwd_fp8(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
        float(q_descale), float(k_descale), float(v_descale), int(bool(causal)), _ptr(workspace),
        nbytes, _stream(stream)))


def forward_fp8(q, k, v, q_descale: float = 1.0, k_descale: float = 1.0, v_descale: float = 1.0,
                scale: float | None = None, causal: bool = False, stream=None):
    """Allocate O (bf16), LSE and the workspace and run fa_fwd_fp8."""
    import torch

    B, H, N, d = _shape(q)
    if scale is None:
        scale = d ** -0.5
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    ws = torch.empty(max(fa_fwd_fp8_workspace_bytes(B, H, N, d), 16), dtype=torch.uint8,
                     device=q.device)
    fa_fwd_fp8(q, k, v, o, lse, scale, q_descale, k_descale, v_descale, causal, ws, stream)
    return o, lse


def fa_fwd_fp8_varlen_workspace_bytes(B: int, max_seqlen_k: int, Hkv: int, d: int) -> int:
    return int(load().fa_fwd_fp8_varlen_workspace_bytes(B, max_seqlen_k, Hkv, d))


def fa_fwd_fp8_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                      max_seqlen_k: int, scale: float, q_descale: float, k_descale: float,
                      v_descale: float, causal: bool, workspace, stream=None) -> None:
    """C ``fa_fwd_fp8_varlen``: q [total_q, H, 128], k, v [total_k, Hkv, 128] e4m3 codes (any
    1-byte dtype), o [total_q, H, 128] bf16, lse [H, total_q] fp32 or None, cu_seqlens_* int32
    [B + 1] on the device."""
    _check_tensors(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, workspace)
    for t in (q, k, v):
        if t.element_size() != 1:
            raise ValueError("q, k and v must hold 1-byte e4m3 codes")
    B, total_q, total_k, H, Hkv, d = _varlen_shapes(q, k, cu_seqlens_q, cu_seqlens_k)
    nbytes = workspace.numel() * workspace.element_size()
    check(load().fa_fwd_fp8_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B,
        int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, H, Hkv, d, float(scale),
        float(q_descale), float(k_descale), float(v_descale), int(bool(causal)), _ptr(workspace),
        nbytes, _stream(stream)))


def forward_fp8_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                       q_descale: float = 1.0, k_descale: float = 1.0, v_descale: float = 1.0,
                       scale: float | None = None, causal: bool = False, stream=None):
    """Allocate O (bf16), LSE and the workspace and run fa_fwd_fp8_varlen."""
    import torch

    total_q, H, d = (int(x) for x in q.shape)
    if scale is None:
        scale = d ** -0.5
    B, Hkv = int(cu_seqlens_q.numel()) - 1, int(k.shape[1])
    o = torch.empty((total_q, H, d), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    ws = torch.empty(max(fa_fwd_fp8_varlen_workspace_bytes(B, max_seqlen_k, Hkv, d), 16),
                     dtype=torch.uint8, device=q.device)
    fa_fwd_fp8_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                      scale, q_descale, k_descale, v_descale, causal, ws, stream)
    return o, lse


def fa_causal_block_counts(q_block: int, Br: int, Bc: int, N: int) -> tuple[int, int]:
    """C ``fa_causal_block_counts``: (unmasked blocks, masked diagonal blocks)."""
    nf, nm = ctypes.c_int(), ctypes.c_int()
    check(load().fa_causal_block_counts(q_block, Br, Bc, N, ctypes.byref(nf), ctypes.byref(nm)))
    return nf.value, nm.value


def forward(q, k, v, scale: float | None = None, causal: bool = False, stream=None,
            impl: int = 0):
    """Allocate O ([B,H,N,d], q's dtype) and LSE ([B,H,N] fp32) and run fa_fwd."""
    import torch

    B, H, N, d = _shape(q)
    if scale is None:
        scale = d ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, scale, causal, stream, impl)
    return o, lse


def backward(q, k, v, o, do, lse, scale: float | None = None, causal: bool = False,
             stream=None, impl: int = 0, workspace=None):
    """Allocate dQ, dK, dV (and the workspace unless given) and run fa_bwd."""
    import torch

    B, H, N, d = _shape(q)
    if scale is None:
        scale = d ** -0.5
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                                device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, causal, workspace, stream, impl)
    return dq, dk, dv


# --------------------------------------------------------------------------- packed batches

def _varlen_shapes(q, k, cu_q, cu_k):
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("packed tensors must be [total, heads, d]")
    if cu_q.dtype != _torch_int32() or cu_k.dtype != _torch_int32():
        raise TypeError("cu_seqlens must be int32")
    if cu_q.dim() != 1 or cu_k.dim() != 1 or cu_q.numel() != cu_k.numel() or cu_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be 1-D with B + 1 entries each")
    total_q, H, d = (int(x) for x in q.shape)
    total_k, Hkv = int(k.shape[0]), int(k.shape[1])
    return cu_q.numel() - 1, total_q, total_k, H, Hkv, d


def _torch_int32():
    import torch

    return torch.int32


def _strides_or_none(*ts):
    """(row, head) element strides of packed [rows, heads, d] views, or None when every tensor
    is contiguous (the plain entry points apply).  The d elements of a head must be
    contiguous."""
    if all(t.is_contiguous() for t in ts):
        return None
    vals = []
    for t in ts:
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError("packed views need contiguous head dimensions (stride 1 in d)")
        vals += [int(t.stride(0)), int(t.stride(1))]
    return (ctypes.c_longlong * len(vals))(*vals)


def _check_views(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, scale: float, causal: bool, stream=None) -> None:
    """C ``fa_fwd_varlen``: q, o [total_q, H, d]; k, v [total_k, Hkv, d] (bf16); lse
    [H, total_q] fp32 (or None); cu_seqlens_* int32 [B + 1] on the device.  Views with other
    row / head strides go through ``fa_fwd_varlen_strided``."""
    _check_views(q, k, v, o)
    _check_tensors(lse, cu_seqlens_q, cu_seqlens_k)
    B, total_q, total_k, H, Hkv, d = _varlen_shapes(q, k, cu_seqlens_q, cu_seqlens_k)
    tail = (_ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, int(max_seqlen_q), int(max_seqlen_k),
            total_q, total_k, H, Hkv, d, float(scale), int(bool(causal)), _stream(stream))
    st = _strides_or_none(q, k, v, o)
    if st is None:
        check(load().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), *tail))
    else:
        check(load().fa_fwd_varlen_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), st,
                                           *tail))


def fa_bwd_varlen_workspace_bytes(total_q: int, H: int, d: int) -> int:
    return int(load().fa_bwd_varlen_workspace_bytes(total_q, H, d))


def fa_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k,
                  max_seqlen_q: int, max_seqlen_k: int, scale: float, causal: bool, workspace,
                  stream=None) -> None:
    """C ``fa_bwd_varlen``: writes dq [total_q, H, d], dk, dv [total_k, Hkv, d] in place.
    Views with other row / head strides go through ``fa_bwd_varlen_strided``."""
    _check_views(q, k, v, o, do, dq, dk, dv)
    _check_tensors(lse, workspace, cu_seqlens_q, cu_seqlens_k)
    B, total_q, total_k, H, Hkv, d = _varlen_shapes(q, k, cu_seqlens_q, cu_seqlens_k)
    nbytes = workspace.numel() * workspace.element_size()
    head = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv))
    tail = (_ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, int(max_seqlen_q), int(max_seqlen_k),
            total_q, total_k, H, Hkv, d, float(scale), int(bool(causal)), _ptr(workspace), nbytes,
            _stream(stream))
    st = _strides_or_none(q, k, v, o, do, dq, dk, dv)
    if st is None:
        check(load().fa_bwd_varlen(*head, *tail))
    else:
        check(load().fa_bwd_varlen_strided(*head, st, *tail))


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                   scale: float | None = None, causal: bool = False, stream=None):
    """Allocate O ([total_q, H, d]) and LSE ([H, total_q] fp32) and run fa_fwd_varlen."""
    import torch

    d = int(q.shape[-1])
    if scale is None:
        scale = d ** -0.5
    o = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    lse = torch.empty((int(q.shape[1]), int(q.shape[0])), dtype=torch.float32, device=q.device)
    fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale,
                  causal, stream)
    return o, lse


def backward_varlen(q, k, v, o, do, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                    max_seqlen_k: int, scale: float | None = None, causal: bool = False,
                    stream=None, workspace=None):
    """Allocate dQ, dK, dV (and the workspace unless given) and run fa_bwd_varlen."""
    import torch

    total_q, H, d = (int(x) for x in q.shape)
    if scale is None:
        scale = d ** -0.5
    if workspace is None:
        workspace = torch.empty(fa_bwd_varlen_workspace_bytes(total_q, H, d), dtype=torch.uint8,
                                device=q.device)
    dq, dk, dv = (torch.empty(t.shape, dtype=t.dtype, device=t.device) for t in (q, k, v))
    fa_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                  max_seqlen_k, scale, causal, workspace, stream)
    return dq, dk, dv


# --------------------------------------------------------------------------- split-KV decode

def fa_decode_num_splits(B: int, Hkv: int, max_seqlen_k: int) -> int:
    """C ``fa_decode_num_splits``: a split count that fills this GPU's SMs."""
    n = int(load().fa_decode_num_splits(B, Hkv, max_seqlen_k))
    check(min(n, 0))
    return n


def fa_decode_workspace_bytes(total_q: int, H: int, d: int, num_splits: int) -> int:
    return int(load().fa_decode_workspace_bytes(total_q, H, d, num_splits))


def fa_fwd_decode(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, scale: float, causal: bool, num_splits: int, workspace,
                  stream=None) -> None:
    """C ``fa_fwd_decode``: packed tensors as fa_fwd_varlen; workspace may be None for
    num_splits = 1."""
    _check_tensors(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, workspace)
    B, total_q, total_k, H, Hkv, d = _varlen_shapes(q, k, cu_seqlens_q, cu_seqlens_k)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(load().fa_fwd_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B,
        int(max_seqlen_q), int(max_seqlen_k), total_q, total_k, H, Hkv, d, float(scale),
        int(bool(causal)), int(num_splits), _ptr(workspace), nbytes, _stream(stream)))


def forward_decode(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                   scale: float | None = None, causal: bool = False, num_splits: int | None = None,
                   stream=None):
    """Allocate O, LSE (and the split workspace) and run fa_fwd_decode."""
    import torch

    total_q, H, d = (int(x) for x in q.shape)
    if scale is None:
        scale = d ** -0.5
    if num_splits is None:
        num_splits = fa_decode_num_splits(int(cu_seqlens_q.numel()) - 1, int(k.shape[1]),
                                          max_seqlen_k)
    nbytes = fa_decode_workspace_bytes(total_q, H, d, num_splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
    o = torch.empty_like(q)
    lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    fa_fwd_decode(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale,
                  causal, num_splits, ws, stream)
    return o, lse
