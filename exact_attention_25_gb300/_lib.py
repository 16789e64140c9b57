"""ctypes binding of libfa.so.  Argument marshalling only: every step of the computation runs
in the library's CUDA kernels.  Tensors are torch CUDA tensors (torch supplies device memory
and streams); shapes are [B, H, N, d] (or, for the variable-length calls, packed
[total, heads, d]), contiguous.  Raises if the library is missing: there
is no fallback implementation."""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")
LIB_CHECKED_PATH = os.path.join(PKG, "libfa_checked.so")

FA_BF16, FA_F32 = 0, 1
STATUS = {
    0: "FA_OK", -1: "FA_ERR_INVALID_ARG", -2: "FA_ERR_UNSUPPORTED_D", -3: "FA_ERR_MISALIGNED",
    -4: "FA_ERR_WORKSPACE", -5: "FA_ERR_LAUNCH", -6: "FA_ERR_DEVICE_TIMEOUT",
    -7: "FA_ERR_TOO_LARGE", -8: "FA_ERR_UNSUPPORTED_DEVICE", -9: "FA_ERR_OUT_OF_BOUNDS",
}
# Every symbol include/fa.h declares (tests check the library exports all of them).
EXPORTS = (
    "fa_fwd", "fa_bwd_workspace_bytes", "fa_bwd", "fa_bwd_stage", "fa_fwd_impl", "fa_bwd_impl",
    "fa_bwd_noalloc", "fa_debug_set_flags",
    "fa_device_status", "fa_set_wait_limit_ns", "fa_status_string", "fa_last_error",
    "fa_causal_block_counts", "fa_version", "fa_fwd_varlen", "fa_bwd_varlen_workspace_bytes",
    "fa_bwd_varlen", "fa_fwd_decode", "fa_decode_workspace_bytes", "fa_decode_num_splits",
    "fa_fwd_varlen_strided", "fa_bwd_varlen_strided", "fa_fwd_gqa", "fa_bwd_gqa",
    "fa_checked_build", "fa_fwd_fp8", "fa_fwd_fp8_workspace_bytes", "fa_fwd_fp8_varlen",
    "fa_fwd_fp8_varlen_workspace_bytes", "fa_tile_order", "fa_order_group", "fa_decode_splits_for",
)

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{STATUS.get(code, code)}: {what}")
        self.code = code


def default_path() -> str:
    """libfa.so, or the bounds-checked libfa_checked.so when the environment sets
    FA_CHECKED=1 (every call then reports out-of-range accesses through fa_device_status)."""
    return LIB_CHECKED_PATH if os.environ.get("FA_CHECKED") == "1" else LIB_PATH


def load(path: str | None = None):
    """Load the library (built by ``exact_attention_25_gb300.build``; see default_path);
    raise if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or default_path()
        if not os.path.exists(p):
            raise FileNotFoundError(
                f"{p} is missing: build it with exact_attention_25_gb300.build.build() "
                "(there is no fallback implementation)")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.fa_fwd_impl.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp]
        lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_bytes.restype = sz
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
        lib.fa_bwd_impl.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp,
                                    sz, i, vp]
        lib.fa_bwd_stage.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp,
                                     sz, i, vp]
        lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.fa_bwd_noalloc.restype = ctypes.c_int
        lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
        lib.fa_bwd_varlen_workspace_bytes.argtypes = [i, i, i]
        lib.fa_bwd_varlen_workspace_bytes.restype = sz
        lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                      i, i, f, i, vp, sz, vp]
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp,
                                   sz, vp]
        lib.fa_fwd_varlen_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                              i, i, f, i, vp]
        lib.fa_bwd_varlen_strided.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i,
                                              i, i, i, i, i, i, i, f, i, vp, sz, vp]
        lib.fa_fwd_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, i,
                                      vp, sz, vp]
        lib.fa_decode_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_decode_workspace_bytes.restype = sz
        lib.fa_decode_num_splits.argtypes = [i, i, i]
        lib.fa_device_status.argtypes = [vp]
        lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.fa_set_wait_limit_ns.restype = None
        lib.fa_debug_set_flags.argtypes = [i]
        lib.fa_debug_set_flags.restype = None
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_last_error.argtypes = []
        lib.fa_last_error.restype = ctypes.c_char_p
        lib.fa_causal_block_counts.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.fa_version.restype = ctypes.c_char_p
        lib.fa_tile_order.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.fa_tile_order.restype = ctypes.c_int
        lib.fa_order_group.argtypes = [i, i, i]
        lib.fa_order_group.restype = ctypes.c_int
        lib.fa_decode_splits_for.argtypes = [i, i, i, i]
        lib.fa_decode_splits_for.restype = ctypes.c_int
        lib.fa_checked_build.argtypes = []
        lib.fa_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_fwd_fp8_workspace_bytes.restype = sz
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, f, f, f, i, vp, sz, vp]
        lib.fa_fwd_fp8_varlen_workspace_bytes.argtypes = [i, i, i, i]
        lib.fa_fwd_fp8_varlen_workspace_bytes.restype = sz
        lib.fa_fwd_fp8_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, f,
                                          f, f, i, vp, sz, vp]
        for fn in ("fa_fwd", "fa_fwd_impl", "fa_bwd", "fa_bwd_impl", "fa_bwd_stage", "fa_device_status",
                   "fa_causal_block_counts", "fa_fwd_varlen", "fa_bwd_varlen", "fa_fwd_decode",
                   "fa_decode_num_splits", "fa_fwd_varlen_strided", "fa_bwd_varlen_strided",
                   "fa_fwd_gqa", "fa_bwd_gqa", "fa_checked_build", "fa_fwd_fp8",
                   "fa_fwd_fp8_varlen"):
            getattr(lib, fn).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


@contextlib.contextmanager
def library(path: str):
    """Route every binding call to the library at ``path`` (for example the checked build)
    inside the ``with`` block; the library in use before is restored on exit."""
    global _lib
    lib = load(path)
    with _lock:
        prev, _lib = _lib, lib
    try:
        yield lib
    finally:
        with _lock:
            _lib = prev


def check(rc: int) -> None:
    if rc != 0:
        raise FaError(rc, load().fa_last_error().decode())


def last_error() -> str:
    return load().fa_last_error().decode()
