"""Seeded synthetic inputs and the named workloads.  Random numbers and shapes only: this
module holds none of the attention arithmetic, so both the library's tests/benchmark and the
oracle can draw their inputs from it.

Recipe (every workload): a CPU ``torch.Generator`` seeded with ``seed`` draws float32
standard-normal tensors shaped [B, H, N, d] in the order Q, K, V, then (if the workload asks
for it) the index set of "hot" query rows, then dO, then the sampled (head, row) pairs.
Multiplicative factors are applied in float32 before the cast to the workload dtype
(round-to-nearest-even for bfloat16).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "bf16" or "fp32"
    causal: bool
    fwd: bool = True
    bwd: bool = False
    in_scale: float = 1.0         # multiplies Q, K, V
    hot_rows_frac: float = 0.0    # fraction of query rows multiplied by hot_rows_mult
    hot_rows_mult: float = 1.0
    n_samples: int = 0            # (head, query-row) samples for oracle checks at full size

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def fwd_flops(self) -> float:
        """4 B H N^2 d, halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f * 0.5 if self.causal else f

    def bwd_flops(self) -> float:
        """2.5 x the forward count."""
        return 2.5 * self.fwd_flops()


WORKLOADS = {
    w.name: w
    for w in (
        Workload("fp32_b1h1_n512_d64", 1, 1, 512, 64, "fp32", False),
        Workload("bf16_b4h16_n4096_d64_hotrows", 4, 16, 4096, 64, "bf16", False,
                 hot_rows_frac=0.01, hot_rows_mult=10.0),
        Workload("bf16_b2h32_n8192_d128_causal", 2, 32, 8192, 128, "bf16", True, in_scale=0.5),
        Workload("bf16_b4h16_n4096_d128_causal_bwd", 4, 16, 4096, 128, "bf16", True, fwd=True,
                 bwd=True),
        Workload("bf16_b1h32_n32000_d128_causal_fwdbwd", 1, 32, 32000, 128, "bf16", True,
                 fwd=True, bwd=True, n_samples=64),
    )
}
# Order of the five workloads of the problem statement.
WORKLOAD_ORDER = list(WORKLOADS)


def generate(w: Workload, seed: int = 0, need_grad_out: bool | None = None) -> dict:
    """Seeded CPU tensors for workload ``w``: q, k, v (w's dtype), do (if backward),
    hot_rows (flattened (b,h,i) indices), samples (list of (h, i))."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (w.B, w.H, w.N, w.d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.in_scale != 1.0:
        q.mul_(w.in_scale)
        k.mul_(w.in_scale)
        v.mul_(w.in_scale)
    hot = None
    if w.hot_rows_frac > 0:
        rows = w.B * w.H * w.N
        hot = torch.randperm(rows, generator=g)[: int(round(w.hot_rows_frac * rows))]
        q.view(rows, w.d)[hot] *= w.hot_rows_mult
    out = {"q": q.to(w.torch_dtype), "k": k.to(w.torch_dtype), "v": v.to(w.torch_dtype),
           "hot_rows": hot}
    if need_grad_out if need_grad_out is not None else w.bwd:
        out["do"] = torch.randn(shape, generator=g, dtype=torch.float32).to(w.torch_dtype)
    if w.n_samples:
        hs = torch.randint(0, w.H, (w.n_samples,), generator=g)
        ids = torch.randint(0, w.N, (w.n_samples,), generator=g)
        out["samples"] = [(int(h), int(i)) for h, i in zip(hs, ids)]
    return out


def random_qkv(B: int, H: int, N: int, d: int, dtype=torch.bfloat16, seed: int = 0,
               in_scale: float = 1.0, with_do: bool = True) -> dict:
    """Seeded standard-normal q, k, v (and do) for ad-hoc shapes (tail sweeps, edge cases)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, d)
    out = {n: (torch.randn(shape, generator=g) * in_scale).to(dtype) for n in ("q", "k", "v")}
    if with_do:
        out["do"] = torch.randn(shape, generator=g).to(dtype)
    return out


def random_varlen(lens_q, lens_k, H: int, Hkv: int, d: int, dtype=torch.bfloat16, seed: int = 0,
                  in_scale: float = 1.0, with_do: bool = True) -> dict:
    """Seeded packed batch: q (and do) [total_q, H, d], k, v [total_k, Hkv, d] standard normal
    (drawn in the order q, k, v, do), and the int32 offsets cu_q, cu_k ([B + 1], CPU) of the
    sequence lengths ``lens_q`` / ``lens_k``."""
    if len(lens_q) != len(lens_k):
        raise ValueError("one query length and one key length per sequence")
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    cu_q = torch.tensor([0] + list(lens_q), dtype=torch.int64).cumsum(0).to(torch.int32)
    cu_k = torch.tensor([0] + list(lens_k), dtype=torch.int64).cumsum(0).to(torch.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    out = {"q": (torch.randn((tq, H, d), generator=g) * in_scale).to(dtype),
           "k": (torch.randn((tk, Hkv, d), generator=g) * in_scale).to(dtype),
           "v": (torch.randn((tk, Hkv, d), generator=g) * in_scale).to(dtype),
           "cu_q": cu_q, "cu_k": cu_k,
           "max_q": max(lens_q), "max_k": max(lens_k)}
    if with_do:
        out["do"] = torch.randn((tq, H, d), generator=g).to(dtype)
    return out


def random_fp8(B: int, H: int, N: int, d: int, seed: int = 0, in_scale: float = 1.0,
               kind: str = "normal") -> dict:
    """Seeded e4m3 inputs (torch.float8_e4m3fn, CPU) with per-tensor descale factors.

    kind "normal": float32 standard-normal Q, K, V times ``in_scale`` (drawn in that order),
    each divided by its descale factor amax / 448 so that its largest magnitude maps to the
    largest e4m3 value, then cast (round to nearest even).
    kind "integer": Q and K rows with at most four entries of +-1 at random positions (the
    rest 0), so every score Q K^T is an integer in [-4, 4]; V as for "normal"; descale
    factors 1 for Q and K.  With the softmax scale ln 2 the weights are powers of two."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, N, d)
    out = {}

    def quantize(x):
        amax = float(x.abs().max())
        ds = amax / 448.0 if amax > 0 else 1.0
        return (x / ds).to(torch.float8_e4m3fn), ds

    if kind == "normal":
        for n in ("q", "k", "v"):
            out[n], out[n + "_descale"] = quantize(torch.randn(shape, generator=g) * in_scale)
    elif kind == "integer":
        for n in ("q", "k"):
            x = torch.zeros(shape)
            cols = torch.randint(0, d, (B, H, N, 4), generator=g)
            signs = torch.randint(0, 3, (B, H, N, 4), generator=g).float() - 1.0  # -1, 0, +1
            x.scatter_(3, cols, signs)  # repeated columns keep one of their values
            out[n], out[n + "_descale"] = x.to(torch.float8_e4m3fn), 1.0
        out["v"], out["v_descale"] = quantize(torch.randn(shape, generator=g) * in_scale)
    else:
        raise ValueError(f"unknown kind {kind!r}")
    return out


def random_fp8_varlen(lens_q, lens_k, H: int, Hkv: int, d: int, seed: int = 0,
                      in_scale: float = 1.0, kind: str = "normal") -> dict:
    """Packed e4m3 batch: q [total_q, H, d], k and v [total_k, Hkv, d] drawn and quantised as
    in random_fp8 (kind "normal" or "integer"), with the int32 offsets cu_q, cu_k ([B + 1],
    CPU) of the sequence lengths ``lens_q`` / ``lens_k``."""
    if len(lens_q) != len(lens_k):
        raise ValueError("one query length and one key length per sequence")
    cu_q = torch.tensor([0] + list(lens_q), dtype=torch.int64).cumsum(0).to(torch.int32)
    cu_k = torch.tensor([0] + list(lens_k), dtype=torch.int64).cumsum(0).to(torch.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    xq = random_fp8(1, 1, tq * H, d, seed=seed, in_scale=in_scale, kind=kind)
    xk = random_fp8(1, 1, tk * Hkv, d, seed=seed + 1, in_scale=in_scale, kind=kind)
    out = {"q": xq["q"].reshape(tq, H, d), "q_descale": xq["q_descale"],
           "k": xk["k"].reshape(tk, Hkv, d), "k_descale": xk["k_descale"],
           "v": xk["v"].reshape(tk, Hkv, d), "v_descale": xk["v_descale"],
           "cu_q": cu_q, "cu_k": cu_k, "max_q": max(lens_q), "max_k": max(lens_k)}
    return out
