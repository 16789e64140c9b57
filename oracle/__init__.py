"""fp64 CPU oracle for exact attention: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The library under test never imports it, and it imports nothing from
the library.  The arithmetic lives in ``oracle.c`` (plain C, fp64); this module only builds
that file with gcc, marshals numpy arrays into it and splits work across host threads.

Every function takes arrays shaped ``[B, H, N, d]`` (``[N, d]`` for the ``*_head`` forms,
packed ``[total, heads, d]`` for ``attention_varlen``), upcasts them exactly to float64 and
returns float64 arrays.  ``lse`` is the natural-log log-sum-exp of the scaled logits, shaped
``[B, H, N]`` (``[H, total_q]`` for ``attention_varlen``).

Parity status of each function (which checks pin it) is listed in the tests
``tests/test_oracle_pins.py``; every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_attention_fwd_head.argtypes = [i, i, d, i, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.oracle_attention_bwd_head.argtypes = [i, i, d, i, _dp, _dp, _dp, _dp, _dp, _dp,
                                                      _dp, _dp, _dp, _dp]
            lib.oracle_attention_fwd_tiled_head.argtypes = [i, i, d, i, i, i, _dp, _dp, _dp, _dp,
                                                            _dp]
            lib.oracle_attention_rows_head.argtypes = [i, i, d, i, _dp, _dp, _dp, _dp, i, _ip,
                                                       _dp, _dp, _dp, _dp, i, _ip, _dp, _dp, i]
            lib.oracle_attention_fwd.argtypes = [i, i, i, d, i, _dp, _dp, _dp, _dp, _dp, i]
            lib.oracle_attention_bwd.argtypes = [i, i, i, d, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                                 _dp, _dp, _dp, i]
            lib.oracle_attention_rect_head.argtypes = [i, i, i, d, i, _dp, _dp, _dp, _dp, _dp,
                                                       _dp, _dp, _dp, _dp, _dp]
            for f in (lib.oracle_attention_fwd_head, lib.oracle_attention_bwd_head,
                      lib.oracle_attention_rect_head,
                      lib.oracle_attention_fwd_tiled_head, lib.oracle_attention_rows_head,
                      lib.oracle_attention_fwd, lib.oracle_attention_bwd):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor: exact upcast on the host
        import torch

        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_dp)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def attention_fwd(q, k, v, scale: float, causal: bool, nthreads: int | None = None):
    """Algorithm 0 over every head: returns (O [B,H,N,d], lse [B,H,N]) in float64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attention_fwd(B * H, N, d, float(scale), int(bool(causal)), _p(q), _p(k),
                                      _p(v), _p(o), _p(lse), nthreads or default_threads())
    _check(rc, "fwd")
    return o, lse


def attention_bwd(q, k, v, do, scale: float, causal: bool, nthreads: int | None = None):
    """Backward over every head: returns dict with dq, dk, dv, o, lse, delta (float64)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    out = {n: np.empty_like(q) for n in ("dq", "dk", "dv", "o")}
    out["lse"] = np.empty((B, H, N), dtype=np.float64)
    out["delta"] = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attention_bwd(
        B * H, N, d, float(scale), int(bool(causal)), _p(q), _p(k), _p(v), _p(do), _p(out["dq"]),
        _p(out["dk"]), _p(out["dv"]), _p(out["o"]), _p(out["lse"]), _p(out["delta"]),
        nthreads or default_threads())
    _check(rc, "bwd")
    return out


def attention_fwd_head(q, k, v, scale: float, causal: bool, want_p: bool = False):
    """Algorithm 0 on one head [N, d]; returns (O, lse) or (O, lse, P)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    o = np.empty_like(q)
    lse = np.empty(N, dtype=np.float64)
    P = np.empty((N, N), dtype=np.float64) if want_p else None
    _check(_load().oracle_attention_fwd_head(N, d, float(scale), int(bool(causal)), _p(q), _p(k),
                                             _p(v), _p(o), _p(lse), _p(P)), "fwd_head")
    return (o, lse, P) if want_p else (o, lse)


def attention_bwd_head(q, k, v, do, scale: float, causal: bool):
    """Backward on one head [N, d]; returns dict dq, dk, dv, o, lse, delta."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    N, d = q.shape
    out = {n: np.empty_like(q) for n in ("dq", "dk", "dv", "o")}
    out["lse"] = np.empty(N, dtype=np.float64)
    out["delta"] = np.empty(N, dtype=np.float64)
    _check(_load().oracle_attention_bwd_head(
        N, d, float(scale), int(bool(causal)), _p(q), _p(k), _p(v), _p(do), _p(out["dq"]),
        _p(out["dk"]), _p(out["dv"]), _p(out["o"]), _p(out["lse"]), _p(out["delta"])), "bwd_head")
    return out


def attention_fwd_tiled_head(q, k, v, scale: float, causal: bool, Br: int, Bc: int):
    """Algorithm 1 (K/V-outer tiled online softmax) on one head; returns (O, lse)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    o = np.empty_like(q)
    lse = np.empty(N, dtype=np.float64)
    _check(_load().oracle_attention_fwd_tiled_head(N, d, float(scale), int(bool(causal)), int(Br),
                                                   int(Bc), _p(q), _p(k), _p(v), _p(o), _p(lse)),
           "fwd_tiled_head")
    return o, lse


def attention_rows_head(q, k, v, do, scale: float, causal: bool, qrows, krows,
                        nthreads: int | None = None):
    """Sampled rows of one head [N, d] without materialising N x N.

    Returns dict: o, lse, delta, dq for each row in ``qrows``; dk, dv for each row in ``krows``.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    N, d = q.shape
    qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int32).reshape(-1))
    kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int32).reshape(-1))
    nq, nk = len(qr), len(kr)
    out = {
        "o": np.empty((nq, d)), "lse": np.empty(nq), "delta": np.empty(nq), "dq": np.empty((nq, d)),
        "dk": np.empty((nk, d)), "dv": np.empty((nk, d)),
    }
    _check(_load().oracle_attention_rows_head(
        N, d, float(scale), int(bool(causal)), _p(q), _p(k), _p(v), _p(do), nq,
        qr.ctypes.data_as(_ip), _p(out["o"]), _p(out["lse"]), _p(out["delta"]), _p(out["dq"]), nk,
        kr.ctypes.data_as(_ip), _p(out["dk"]), _p(out["dv"]), nthreads or default_threads()),
        "rows_head")
    return out


def attention_rect_head(q, k, v, scale: float, causal: bool, do=None):
    """One head with Nq query rows [Nq, d] and Nk key rows [Nk, d]; causal is aligned to the
    bottom-right corner (key j visible to query i iff j <= i + Nk - Nq).  Returns dict o, lse
    (and, with do, delta, dq, dk, dv)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Nq, d = q.shape
    Nk = k.shape[0]
    out = {"o": np.empty((Nq, d)), "lse": np.empty(Nq)}
    if do is not None:
        do = _f64(do)
        out |= {"delta": np.empty(Nq), "dq": np.empty((Nq, d)), "dk": np.empty((Nk, d)),
                "dv": np.empty((Nk, d))}
    g = out.get
    _check(_load().oracle_attention_rect_head(
        Nq, Nk, d, float(scale), int(bool(causal)), _p(q), _p(k), _p(v), _p(do), _p(out["o"]),
        _p(out["lse"]), _p(g("delta")), _p(g("dq")), _p(g("dk")), _p(g("dv"))), "rect_head")
    return out


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool, do=None,
                     nthreads: int | None = None):
    """Packed variable-length batch with grouped key/value heads.

    q (and do) are ``[total_q, H, d]``, k and v ``[total_k, Hkv, d]``; sequence b owns query
    rows ``cu_seqlens_q[b]:cu_seqlens_q[b+1]`` and key rows ``cu_seqlens_k[b]:cu_seqlens_k[b+1]``.
    Query head h attends to key/value head ``h // (H // Hkv)``.  Each (sequence, head) pair is
    one ``attention_rect_head`` problem.  The gradients of a shared key/value head are the sum
    over the query heads that read it (chain rule), added in head order.
    Returns dict o ``[total_q, H, d]``, lse ``[H, total_q]`` and, with do, delta
    ``[H, total_q]``, dq ``[total_q, H, d]``, dk and dv ``[total_k, Hkv, d]``.
    """
    import concurrent.futures as cf

    q, k, v = _f64(q), _f64(k), _f64(v)
    do = None if do is None else _f64(do)
    cu_q = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    total_q, H, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    if H % Hkv or len(cu_q) != len(cu_k):
        raise ValueError("H must be a multiple of Hkv; cu_seqlens must have equal lengths")
    G = H // Hkv
    jobs = [(b, h) for b in range(len(cu_q) - 1) for h in range(H)]

    def one(job):
        b, h = job
        qs, ks = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        hk = h // G
        return attention_rect_head(q[qs, h], k[ks, hk], v[ks, hk], scale, causal,
                                   None if do is None else do[qs, h])

    with cf.ThreadPoolExecutor(max_workers=nthreads or default_threads()) as ex:
        res = list(ex.map(one, jobs))
    out = {"o": np.zeros((total_q, H, d)), "lse": np.zeros((H, total_q))}
    if do is not None:
        out |= {"delta": np.zeros((H, total_q)), "dq": np.zeros((total_q, H, d)),
                "dk": np.zeros((total_k, Hkv, d)), "dv": np.zeros((total_k, Hkv, d))}
    for (b, h), r in zip(jobs, res):
        qs, ks = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        out["o"][qs, h] = r["o"]
        out["lse"][h, qs] = r["lse"]
        if do is not None:
            out["delta"][h, qs] = r["delta"]
            out["dq"][qs, h] = r["dq"]
            out["dk"][ks, h // G] += r["dk"]
            out["dv"][ks, h // G] += r["dv"]
    return out


# --------------------------------------------------------------------------- e4m3 inputs

def e4m3_decode(codes) -> np.ndarray:
    """Value of OCP FP8 E4M3 codes (uint8), from the format's definition: bit 7 the sign,
    bits 6-3 the exponent with bias 7, bits 2-0 the mantissa; exponent field 0 holds the
    subnormals m/8 * 2^-6; the codes S.1111.111 are NaN and there is no infinity, so the
    largest finite value is 1.75 * 2^8 = 448."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


def _codes(t) -> np.ndarray:
    """The bytes of a 1-byte tensor (torch float8 / uint8) or array, as uint8."""
    if hasattr(t, "detach"):
        import torch

        t = t.detach().to("cpu").contiguous().view(torch.uint8).numpy()
    return np.ascontiguousarray(t, dtype=np.uint8)


def attention_fp8(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float,
                  scale: float, causal: bool):
    """Exact attention on the values that e4m3 codes stand for (per-tensor scaling):
    Q = q_descale * e4m3(q8), K = k_descale * e4m3(k8), V = v_descale * e4m3(v8), all
    ``[B, H, N, d]``.  Returns dict o, lse (Algorithm 0 on those values, as attention_fwd_head)
    , ``pv_abs`` = sum_j P_ij |V_jc| (the scale of accumulation error) and ``bound``: per
    element of O, the largest deviation that rounding every probability to
    e4m3 before the P V product can cause when O is divided by the unrounded row sum,
        bound_ic = sum_j max(2^-4 P_ij, 2^-10 max_j' P_ij') |V_jc|   (over the keys row i sees),
    with 2^-4 the relative half-spacing of normal e4m3 values and 2^-10 half the subnormal
    spacing (probabilities held relative to a stale row maximum only scale these terms by a
    factor <= 1, and the row sum is at least 1 / max_j P_ij).  Rounding of O to bf16 comes on
    top."""
    q = e4m3_decode(_codes(q8)) * float(q_descale)
    k = e4m3_decode(_codes(k8)) * float(k_descale)
    v = e4m3_decode(_codes(v8)) * float(v_descale)
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    bound = np.empty((B, H, N, d))
    pv_abs = np.empty((B, H, N, d))
    for b in range(B):
        for h in range(H):
            ob, lb, P = attention_fwd_head(q[b, h], k[b, h], v[b, h], scale, causal, want_p=True)
            seen = np.ones((N, N), dtype=bool)
            if causal:
                seen = np.tril(seen)
            w = np.maximum(P / 16.0, P.max(axis=1, keepdims=True) / 1024.0) * seen
            o[b, h], lse[b, h] = ob, lb
            bound[b, h] = w @ np.abs(v[b, h])
            pv_abs[b, h] = P @ np.abs(v[b, h])
    return {"o": o, "lse": lse, "bound": bound, "pv_abs": pv_abs}


def attention_fp8_rows(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float,
                       scale: float, causal: bool, rows):
    """attention_fp8 for the sampled query rows ``rows`` = [(b, h, i), ...] only, each from its
    own row of scores (Algorithm 0 restricted to that row, causal keys j <= i).  Returns dict
    o [n, d], lse [n], bound [n, d], pv_abs [n, d] in the order of ``rows``."""
    qc, kc, vc = _codes(q8), _codes(k8), _codes(v8)
    out = {"o": [], "lse": [], "bound": [], "pv_abs": []}
    for b, h, i in rows:
        qi = e4m3_decode(qc[b, h, i]) * float(q_descale)
        n = i + 1 if causal else kc.shape[2]
        kk = e4m3_decode(kc[b, h, :n]) * float(k_descale)
        vv = e4m3_decode(vc[b, h, :n]) * float(v_descale)
        s = scale * (kk @ qi)
        m = s.max()
        e = np.exp(s - m)
        tot = e.sum()
        P = e / tot
        out["o"].append(P @ vv)
        out["lse"].append(m + np.log(tot))
        w = np.maximum(P / 16.0, P.max() / 1024.0)
        out["bound"].append(w @ np.abs(vv))
        out["pv_abs"].append(P @ np.abs(vv))
    return {key: np.array(val) for key, val in out.items()}


def attention_fp8_varlen(q8, k8, v8, cu_seqlens_q, cu_seqlens_k, q_descale: float,
                         k_descale: float, v_descale: float, scale: float, causal: bool):
    """attention_fp8 for a packed batch with grouped key/value heads: the sequences, the head
    mapping h -> h // (H // Hkv) and the bottom-right causal mask (query i of a sequence with
    nq queries and nk keys sees key j iff j <= i + nk - nq) of attention_varlen.  Algorithm 0
    per (sequence, head) with S and P materialised in float64; a row that sees no key has
    O = 0, lse = -inf and bound 0.  Returns dict o, bound, pv_abs ``[total_q, H, d]`` and lse
    ``[H, total_q]``."""
    q = e4m3_decode(_codes(q8)) * float(q_descale)
    k = e4m3_decode(_codes(k8)) * float(k_descale)
    v = e4m3_decode(_codes(v8)) * float(v_descale)
    cu_q = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    total_q, H, d = q.shape
    G = H // k.shape[1]
    out = {"o": np.zeros((total_q, H, d)), "lse": np.full((H, total_q), -np.inf),
           "bound": np.zeros((total_q, H, d)), "pv_abs": np.zeros((total_q, H, d))}
    for b in range(len(cu_q) - 1):
        qs, ks = slice(cu_q[b], cu_q[b + 1]), slice(cu_k[b], cu_k[b + 1])
        nq, nk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        if nq == 0 or nk == 0:
            continue
        seen = np.ones((nq, nk), dtype=bool)
        if causal:
            seen = np.arange(nk)[None, :] <= np.arange(nq)[:, None] + (nk - nq)
        live = seen.any(axis=1)
        for h in range(H):
            vv = v[ks, h // G]
            S = np.where(seen, scale * (q[qs, h] @ k[ks, h // G].T), -np.inf)
            m = np.where(live, S.max(axis=1, initial=-np.inf), 0.0)
            e = np.where(seen, np.exp(S - m[:, None]), 0.0)
            tot = e.sum(axis=1)
            P = np.divide(e, tot[:, None], out=np.zeros_like(e), where=live[:, None])
            w = np.maximum(P / 16.0, P.max(axis=1, keepdims=True) / 1024.0) * seen
            rows = np.arange(cu_q[b], cu_q[b + 1])
            out["o"][rows, h] = P @ vv
            out["lse"][h, rows] = np.where(live, m + np.log(np.where(live, tot, 1.0)), -np.inf)
            out["bound"][rows, h] = w @ np.abs(vv)
            out["pv_abs"][rows, h] = P @ np.abs(vv)
    return out
